// The gated delta rule with a replay log: in-place decode, ReplaySSM verify
// and commit ("Why Speculative Decoding Slows Hybrid Mamba Models", When the
// layer is a different kind of recurrence: the update must unroll as a decay
// plus a sum, and Gated DeltaNet's does).  Per value head h, key head
// g(h) = h / (H / G):
//   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t
// with S fp32 [dv][dk].
//
// Every kernel here is bound by the state's bytes, and the state's rows are
// independent: with the token's k, q and scalars fixed, row p of S_t depends
// only on row p of S_{t-1} (w = S[p] . k, S[p] <- exp(g) S[p] + (beta v[p] -
// exp(g) beta w) k), and row p of an output is S[p] . q.  So a warp streams
// four rows at a time, eight lanes a row; lane s of a row holds the 16-byte
// pieces n = 4 (s + 8 i) .. + 3 (i < dk / 32), so that each load instruction
// of the warp covers four whole 128-byte lines, and a row's dot products take
// three shuffles.
//
// Replay verify (The Fix: outputs from the checkpoint and the log, no state
// written) unrolls the output at position m (the log's K tokens, then the
// step tokens) as o_m = S_ckpt u_0 + sum_i beta_i (k_i . u_i) v_i, where
// u_m = q_m and u_{i-1} = exp(g_i) (u_i - beta_i k_i (k_i . u_i)).  A
// coefficient kernel walks those sweeps (a dk-vector per step token, on eight
// lanes each), forms the log terms sum_i beta_i (k_i . u_i) v_i and stages the
// step after the log; a streaming kernel then reads each checkpoint row once
// for all step tokens.
#include <algorithm>
#include <type_traits>
#include <utility>
#include <cstring>
#include <vector>

#include "ssm_gdn.h"
#include "ssm_internal.cuh"
#include "tc.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kGdnMaxBatch = 1024;  // requests per launch: slot lists travel in kernel parameters
constexpr int kGdnListCount = 4 * kGdnMaxBatch;  // the fold list's count, after its {request, slot, M, 0} entries
constexpr int kGdnWarps = 8;
constexpr int kGdnThreads = 32 * kGdnWarps;
constexpr int kGdnMaxWindow = 32, kGdnMaxTokens = 32;

struct GdnArgs {
    float *state;
    void *log_k, *log_v;  // [slot][wcap][G][dk], [slot][wcap][H][dv], input dtype
    float *log_g, *log_b; // [slot][wcap][H]
    int32_t *log_len;
    int64_t *position;
    uint32_t *slot_flags, *flags;
    float *uq, *lt;       // verify scratch: [request][H][t1max][dk] queries, [request][H][t1max][dv] log terms
    int uq_nm;            // 0: uq as above; else uq_rows rows per (request, head) in the tensor-core
    int uq_rows;          // kernel's operand layout: [4 blocks of 32 columns][uq_nm rows][32], 16-byte chunk c
                          // of row j at c ^ (j % 8)
    int32_t *fold_m;      // commit: tokens to fold per request of the launch (0: none)
    int32_t *fold_list;   // commit: the launch's folding requests {i, slot, M, 0}, their count at [kGdnListCount]
    const void *q, *k, *v;
    const float *g, *beta;
    void *y;
    const int32_t *accept;
    int H, G, hpg, dv, W, wcap, t1max, n_tok, batch, force_fold;
    int32_t slots[kGdnMaxBatch];
    int32_t ntok[kGdnMaxBatch];
};

__device__ __forceinline__ float red8(float v) {  // sum over the eight lanes of a row
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// x . y accumulated in a pair of partial sums with the two-wide FMA (half the instructions)
__device__ __forceinline__ float2 dot4x2(float4 x, float4 y, float2 acc) {
    acc = ffma2(make_float2(x.x, x.y), make_float2(y.x, y.y), acc);
    return ffma2(make_float2(x.z, x.w), make_float2(y.z, y.w), acc);
}

// x + c k with the two-wide FMA
__device__ __forceinline__ float4 add_ck4(float4 x, float c, float4 k) {
    const float2 lo = ffma2(make_float2(c, c), make_float2(k.x, k.y), make_float2(x.x, x.y));
    const float2 hi = ffma2(make_float2(c, c), make_float2(k.z, k.w), make_float2(x.z, x.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ float4 scale4(float c, float4 x) {
    const float2 lo = ffma2(make_float2(c, c), make_float2(x.x, x.y), make_float2(0.f, 0.f));
    const float2 hi = ffma2(make_float2(c, c), make_float2(x.z, x.w), make_float2(0.f, 0.f));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ float4 axpy4(float al, float4 x, float c, float4 k) {  // al x + c k
    return make_float4(fmaf(al, x.x, c * k.x), fmaf(al, x.y, c * k.y), fmaf(al, x.z, c * k.z),
                       fmaf(al, x.w, c * k.w));
}

// rows x cols values (cols a multiple of 4) of a strided global matrix into fp32 shared memory
// [rows][cols]: four values a load and four loads in flight per thread, since a CTA's staging is
// otherwise a chain of round trips to memory.  Returns true if a value is not finite.
template <typename TI>
__device__ __forceinline__ bool stage_rows(float *dst, const TI *src, size_t stride, int rows, int cols, int tid,
                                           int nthr) {
    const int cq = cols >> 2, total = rows * cq;
    bool bad = false;
    for (int base = tid; base < total; base += 4 * nthr) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = base + u * nthr;
            if (e < total) {
                const int r = e / cq, c = e - r * cq;
                v[u] = load4(src + (size_t)r * stride, (size_t)4 * c);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = base + u * nthr;
            if (e < total) {
                const int r = e / cq, c = e - r * cq;
                bad |= !finite4(v[u]);
                *reinterpret_cast<float4 *>(dst + (size_t)r * cols + 4 * c) = v[u];
            }
        }
    }
    return bad;
}

// Four values of the input type as one load, and whether one of them is not finite (all exponent bits set).
template <typename TI> struct Vec4;
template <> struct Vec4<float> {
    using T = uint4;
    __device__ static bool bad(T v) {
        return ((v.x & 0x7F800000u) == 0x7F800000u) | ((v.y & 0x7F800000u) == 0x7F800000u) |
               ((v.z & 0x7F800000u) == 0x7F800000u) | ((v.w & 0x7F800000u) == 0x7F800000u);
    }
};
template <> struct Vec4<__nv_bfloat16> {
    using T = uint2;
    __device__ static bool bad(T v) {
        return ((v.x & 0x7F80u) == 0x7F80u) | ((v.x & 0x7F800000u) == 0x7F800000u) | ((v.y & 0x7F80u) == 0x7F80u) |
               ((v.y & 0x7F800000u) == 0x7F800000u);
    }
};

__device__ __forceinline__ void poison(const GdnArgs &a, int slot, uint32_t flag) {
    atomicOr(a.flags, flag);
    atomicOr(a.slot_flags + slot, kSlotPoisoned);
}

// A warp holds kRG groups of four rows at once (rows p0 + 32 kGdnWarps... apart), so that 8 KiB of
// loads are in flight per warp; rows past dv are skipped (dv is a multiple of 4: a group is whole or
// absent).
constexpr int kRG = 4;

template <int NV>
__device__ __forceinline__ void load_rows(const float *st, int DK, int dv, int p0, int r, int s, int (&pr)[kRG],
                                          bool (&ok)[kRG], float4 (&sv)[kRG][NV]) {
#pragma unroll
    for (int q = 0; q < kRG; ++q) {
        pr[q] = p0 + 4 * kGdnWarps * q + r;
        ok[q] = pr[q] < dv;
    }
#pragma unroll
    for (int q = 0; q < kRG; ++q)
#pragma unroll
        for (int e = 0; e < NV; ++e)
            sv[q][e] = ok[q] ? ld_stream(st + (size_t)pr[q] * DK + 4 * (s + 8 * e)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int NV>
__device__ __forceinline__ void store_rows(float *st, int DK, const int (&pr)[kRG], const bool (&ok)[kRG], int s,
                                           const float4 (&sv)[kRG][NV]) {
#pragma unroll
    for (int q = 0; q < kRG; ++q)
        if (ok[q])
#pragma unroll
            for (int e = 0; e < NV; ++e) st_stream(st + (size_t)pr[q] * DK + 4 * (s + 8 * e), sv[q][e]);
}

// ---------------------------------------------------------------------------- decode

// One token per request, in place.  Grid (H, batch).
template <int DK, typename TI>
__global__ void __launch_bounds__(kGdnThreads, 2) gdn_decode_kernel(const __grid_constant__ GdnArgs a) {
    constexpr int NV = DK / 32;
    __shared__ __align__(16) float sk[DK], sq[DK];
    const int h = blockIdx.x, i = blockIdx.y, slot = a.slots[i], kh = h / a.hpg;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 3, s = lane & 7;
    if (a.slot_flags[slot] & kSlotPoisoned) {
        if (tid == 0) atomicOr(a.flags, SSM_FLAG_POISONED_SLOT);
        return;
    }
    if (a.log_len[slot] != 0) {  // the state in place is the checkpoint: tokens in the log would be lost
        if (tid == 0) poison(a, slot, SSM_FLAG_LOG_NOT_EMPTY);
        return;
    }
    float *st = a.state + ((size_t)slot * a.H + h) * a.dv * DK;
    // the warp's first rows are in flight while the token is read and checked
    int pr[kRG];
    bool ok[kRG];
    float4 sv[kRG][NV];
    load_rows<NV>(st, DK, a.dv, 4 * warp, r, s, pr, ok, sv);
    const TI *qg = static_cast<const TI *>(a.q) + ((size_t)i * a.G + kh) * DK;
    const TI *kg = static_cast<const TI *>(a.k) + ((size_t)i * a.G + kh) * DK;
    const TI *vh = static_cast<const TI *>(a.v) + ((size_t)i * a.H + h) * a.dv;
    const float gg = a.g[(size_t)i * a.H + h], bb = a.beta[(size_t)i * a.H + h];
    bool bad = !(isfinite(gg) && isfinite(bb));
    for (int n = tid; n < DK; n += kGdnThreads) {
        sk[n] = to_f(kg[n]);
        sq[n] = to_f(qg[n]);
        bad |= !(isfinite(sk[n]) && isfinite(sq[n]));
    }
    for (int p = tid; p < a.dv; p += kGdnThreads) bad |= !isfinite(to_f(vh[p]));
    if (__syncthreads_or(bad)) {
        if (tid == 0) poison(a, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }
    const float alpha = expf(gg), ab = alpha * bb;
    float4 kr[NV];  // q is read from shared memory where it is used (registers go to the rows)
#pragma unroll
    for (int e = 0; e < NV; ++e) kr[e] = *reinterpret_cast<const float4 *>(sk + 4 * (s + 8 * e));
    TI *yh = static_cast<TI *>(a.y) + ((size_t)i * a.H + h) * a.dv;
    for (int p0 = 4 * warp; p0 < a.dv; p0 += 4 * kGdnWarps * kRG) {
        if (p0 != 4 * warp) load_rows<NV>(st, DK, a.dv, p0, r, s, pr, ok, sv);
        float w[kRG];
#pragma unroll
        for (int q = 0; q < kRG; ++q) {
            w[q] = 0.f;
#pragma unroll
            for (int e = 0; e < NV; ++e) w[q] += dot4(sv[q][e], kr[e]);
        }
#pragma unroll
        for (int q = 0; q < kRG; ++q) w[q] = red8(w[q]);
#pragma unroll
        for (int q = 0; q < kRG; ++q) {
            const float c = ok[q] ? bb * to_f(vh[pr[q]]) - ab * w[q] : 0.f;
            float o = 0.f;
#pragma unroll
            for (int e = 0; e < NV; ++e) {
                sv[q][e] = axpy4(alpha, sv[q][e], c, kr[e]);
                o += dot4(sv[q][e], *reinterpret_cast<const float4 *>(sq + 4 * (s + 8 * e)));
            }
            w[q] = o;
        }
#pragma unroll
        for (int q = 0; q < kRG; ++q) w[q] = red8(w[q]);
        store_rows<NV>(st, DK, pr, ok, s, sv);
#pragma unroll
        for (int q = 0; q < kRG; ++q)
            if (s == 0 && ok[q]) yh[pr[q]] = from_f<TI>(w[q]);
    }
    if (h == 0 && tid == 0) a.position[slot] += 1;
}

// ---------------------------------------------------------------------------- replay verify

// The coefficient kernel's shared memory (bytes): for fp32 inputs the keys [wcap][DK] (the log's, then
// the step's), fp32 queries [t1max][DK], exp(g) and beta [hpg][wcap] each, the log-term weights
// [hpg][t1max][wcap], the values [wcap][hpg dv] as given (the log's, then the step's), and for bf16
// inputs the keys and queries as given [wcap + t1max][DK] (the sweeps read those keys directly).
struct CoefLayout {
    size_t sq, sal, sbe, scw, svr, rkq, total;
};
__host__ __device__ inline CoefLayout coef_layout(int DK, int dv, int wcap, int t1max, int hpg, int in_b) {
    CoefLayout L;
    size_t o = in_b == 2 ? 0 : (size_t)wcap * DK * 4;
    L.sq = o;
    o += (size_t)t1max * DK * 4;
    L.sal = o;
    o += (size_t)hpg * wcap * 4;
    L.sbe = o;
    o += (size_t)hpg * wcap * 4;
    L.scw = o;
    o += (size_t)hpg * t1max * wcap * 4;
    o = (o + 15) & ~(size_t)15;
    L.svr = o;
    o += (size_t)wcap * hpg * dv * in_b;
    o = (o + 15) & ~(size_t)15;
    L.rkq = o;
    if (in_b == 2) o += (size_t)(wcap + t1max) * DK * 2;
    L.total = o;
    return L;
}
__host__ __device__ inline size_t gdn_coef_smem(int DK, int dv, int wcap, int t1max, int hpg, int in_b) {
    return coef_layout(DK, dv, wcap, t1max, hpg, in_b).total;
}

// 8-byte asynchronous global -> shared copy (both addresses 8-byte aligned)
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// Two fp32 values rounded to bf16 (round to nearest even) and packed, the first in the low half.
__device__ __forceinline__ uint32_t bf2_pack(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Four values of the input type from shared memory, widened to fp32 (bf16: the bits moved up 16).
__device__ __forceinline__ float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 lds4(const __nv_bfloat16 *p) {
    const uint2 r = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u), __uint_as_float(r.y << 16),
                       __uint_as_float(r.y & 0xFFFF0000u));
}

// Grid (G, batch): one CTA per request and key head, whose logged and step keys serve all its value
// heads.  It checks and stages the step, then walks the sweeps: sweep (value head, step token) takes
// the eight lanes of a row group, u in the rows' layout, so that k_t . u takes three shuffles.  A
// warp's four sweeps run the same number of steps (its longest), the shorter ones idle at the end.
template <int DK, typename TI>
__global__ void __launch_bounds__(kGdnThreads, 4) gdn_coef_kernel(const __grid_constant__ GdnArgs a) {
    constexpr int NV = DK / 32;
    extern __shared__ __align__(16) float gsm[];
    const int kh = blockIdx.x, i = blockIdx.y, slot = a.slots[i], hpg = a.hpg, h0 = kh * hpg;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 3, s = lane & 7;
    const int nthr = blockDim.x, nwarps = nthr >> 5;  // sized by the host to the sweeps
    const int T1 = a.n_tok;
    // the tensor-core streaming kernel may start its checkpoint loads as this grid drains; it waits for
    // this grid's completion before it reads anything written here.  This grid may itself start as the
    // previous commit's fold drains: nothing is read before that grid has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (a.slot_flags[slot] & kSlotPoisoned) {
        if (tid == 0) atomicOr(a.flags, SSM_FLAG_POISONED_SLOT);
        return;
    }
    const int K = a.log_len[slot], m = K + T1, hdv = hpg * a.dv;
    const CoefLayout L = coef_layout(DK, a.dv, a.wcap, a.t1max, hpg, (int)sizeof(TI));
    char *base = reinterpret_cast<char *>(gsm);
    float *sk = gsm;                                       // fp32 inputs: [wcap][DK] the log's keys, then the step's
    float *sq = reinterpret_cast<float *>(base + L.sq);    // [t1max][DK]
    float *sal = reinterpret_cast<float *>(base + L.sal);  // [hpg][wcap] exp(g)
    float *sbe = reinterpret_cast<float *>(base + L.sbe);  // [hpg][wcap] beta
    float *scw = reinterpret_cast<float *>(base + L.scw);  // [hpg][t1max][wcap] the weights of the logged values
    TI *svr = reinterpret_cast<TI *>(base + L.svr);        // [wcap][hpg dv] values as given
    // keys and queries as given: fp32 inputs land in place, bf16 ones beside and are widened below
    constexpr bool kWide = sizeof(TI) == 2;
    TI *rk = kWide ? reinterpret_cast<TI *>(base + L.rkq) : reinterpret_cast<TI *>(sk);
    TI *rq = kWide ? rk + (size_t)a.wcap * DK : reinterpret_cast<TI *>(sq);
    const TI *lk = static_cast<const TI *>(a.log_k) + (size_t)slot * a.wcap * a.G * DK + (size_t)kh * DK;
    const TI *lv = static_cast<const TI *>(a.log_v) + ((size_t)slot * a.wcap * a.H + h0) * a.dv;
    const size_t kstep = ((size_t)i * T1 * a.G + kh) * DK;  // step token 0's key (and query) of this key head
    const TI *ks = static_cast<const TI *>(a.k) + kstep, *qs = static_cast<const TI *>(a.q) + kstep;
    const TI *vs = static_cast<const TI *>(a.v) + ((size_t)i * T1 * a.H + h0) * a.dv;
    const size_t krow = (size_t)a.G * DK, vrow = (size_t)a.H * a.dv;
    // every load of the CTA in flight at once: the keys (the log's, then the step's) and the step's
    // queries in 16-byte pieces, the values of the hpg value heads (one contiguous run a token), then the
    // gates with plain loads while the copies land
    {
        constexpr int KCH = DK * (int)sizeof(TI) / 16;  // pieces of a key row
        for (int c = tid; c < (m + T1) * KCH; c += nthr) {
            const int row = c / KCH, off = (c % KCH) * (16 / (int)sizeof(TI));
            const TI *src = row < K ? lk + (size_t)row * krow
                          : row < m ? ks + (size_t)(row - K) * krow
                                    : qs + (size_t)(row - m) * krow;
            TI *dst = row < m ? rk + (size_t)row * DK : rq + (size_t)(row - m) * DK;
            cp_async16(dst + off, src + off);
        }
        if ((a.dv * (int)sizeof(TI)) % 16 == 0) {  // every head's run starts on a 16-byte boundary
            const int vch = hdv * (int)sizeof(TI) / 16;
            for (int c = tid; c < m * vch; c += nthr) {
                const int row = c / vch, off = (c - row * vch) * (16 / (int)sizeof(TI));
                const TI *src = row < K ? lv + (size_t)row * vrow : vs + (size_t)(row - K) * vrow;
                cp_async16(svr + (size_t)row * hdv + off, src + off);
            }
        } else {  // bf16 with dv = 4 (mod 8): 8-byte pieces
            const int vch = hdv * (int)sizeof(TI) / 8;
            for (int c = tid; c < m * vch; c += nthr) {
                const int row = c / vch, off = (c - row * vch) * (8 / (int)sizeof(TI));
                const TI *src = row < K ? lv + (size_t)row * vrow : vs + (size_t)(row - K) * vrow;
                cp_async8(svr + (size_t)row * hdv + off, src + off);
            }
        }
        cp_async_commit();
    }
    bool bad = false;
    for (int e = tid; e < hpg * m; e += nthr) {
        const int hl = e / m, t = e - hl * m;
        float gv, bv;
        if (t < K) {
            gv = a.log_g[((size_t)slot * a.wcap + t) * a.H + h0 + hl];
            bv = a.log_b[((size_t)slot * a.wcap + t) * a.H + h0 + hl];
        } else {  // the step's, checked and logged after the log (for the commit)
            const size_t src = ((size_t)i * T1 + t - K) * a.H + h0 + hl, dst = ((size_t)slot * a.wcap + t) * a.H + h0 + hl;
            gv = a.g[src];
            bv = a.beta[src];
            bad |= !(isfinite(gv) && isfinite(bv));
            a.log_g[dst] = gv;
            a.log_b[dst] = bv;
        }
        sal[(size_t)hl * a.wcap + t] = expf(gv);
        sbe[(size_t)hl * a.wcap + t] = bv;
    }
    cp_async_wait<0>();
    __syncthreads();
    // widen the keys and queries (bf16), check the step's rows, and copy the step after the log (the
    // positions past log_len: a rejected request leaves nothing behind that a later commit reads)
    using V4 = typename Vec4<TI>::T;
    if constexpr (kWide) {
        // the log's keys were checked when they were logged: the pass starts at the step's keys; the
        // sweeps read bf16 keys as staged, so only the queries are widened
        for (int c = tid; c < (m + T1 - K) * (DK / 4); c += nthr) {
            const int row = K + c / (DK / 4), off = 4 * (c % (DK / 4));
            const TI *src = row < m ? rk + (size_t)row * DK + off : rq + (size_t)(row - m) * DK + off;
            const V4 raw = *reinterpret_cast<const V4 *>(src);
            bad |= Vec4<TI>::bad(raw);
            if (row < m)
                *reinterpret_cast<V4 *>(static_cast<TI *>(a.log_k) + ((size_t)slot * a.wcap + row) * krow +
                                        (size_t)kh * DK + off) = raw;
            else
                *reinterpret_cast<float4 *>(sq + (size_t)(row - m) * DK + off) = lds4(src);
        }
    } else {
        for (int c = tid; c < (m + T1) * (DK / 4); c += nthr) {
            const int row = c / (DK / 4), off = 4 * (c % (DK / 4));
            const TI *src = row < m ? rk + (size_t)row * DK + off : rq + (size_t)(row - m) * DK + off;
            if (row >= K) {
                const V4 raw = *reinterpret_cast<const V4 *>(src);
                bad |= Vec4<TI>::bad(raw);
                if (row < m)
                    *reinterpret_cast<V4 *>(static_cast<TI *>(a.log_k) +
                                            ((size_t)slot * a.wcap + row) * krow + (size_t)kh * DK + off) = raw;
            }
        }
    }
    for (int c = tid; c < T1 * (hdv / 4); c += nthr) {
        const int j = c / (hdv / 4), off = 4 * (c - j * (hdv / 4));
        const V4 raw = *reinterpret_cast<const V4 *>(svr + (size_t)(K + j) * hdv + off);
        bad |= Vec4<TI>::bad(raw);
        *reinterpret_cast<V4 *>(static_cast<TI *>(a.log_v) + ((size_t)slot * a.wcap * a.H + h0) * a.dv +
                                (size_t)(K + j) * vrow + off) = raw;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) poison(a, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }
    // the sweeps: sweep id = 4 * (warp + kGdnWarps * round) + r over hpg * T1 (head hl = id / T1, token j)
    const int nsw = hpg * T1;
    for (int base = 4 * warp; base < nsw; base += 4 * nwarps) {
        const int id = base + r;
        const bool act = id < nsw;
        const int hl = act ? id / T1 : 0, j = act ? id - hl * T1 : 0;
        const int mj = act ? K + j + 1 : 0;
        // the warp's longest sweep: its last active id has the largest j or a later head (then j runs
        // from 0 again), so take the largest of the four
        int mmax = mj;
        mmax = max(mmax, __shfl_xor_sync(0xffffffffu, mmax, 8));
        mmax = max(mmax, __shfl_xor_sync(0xffffffffu, mmax, 16));
        float4 u[NV];
#pragma unroll
        for (int e = 0; e < NV; ++e) u[e] = *reinterpret_cast<const float4 *>(sq + (size_t)j * DK + 4 * (s + 8 * e));
        const float *al = sal + (size_t)hl * a.wcap, *be = sbe + (size_t)hl * a.wcap;
        float *csj = scw + ((size_t)hl * a.t1max + j) * a.wcap;
        // the weight just past the sweep is zero: the log terms below take step tokens in pairs over the
        // longer one's span (mj < wcap whenever a later step token exists)
        if (act && s == 0 && mj < a.wcap) csj[mj] = 0.f;
        // the next step's key is loaded while this step's dot product is reduced; bf16 pools read the keys
        // as given (8-byte pieces, half the shared-memory wavefronts of the fp32 rows) and widen them here
        using KRaw = typename std::conditional<kWide, uint2, float4>::type;
        auto kload = [&](int t, KRaw (&kr)[NV]) {
#pragma unroll
            for (int e = 0; e < NV; ++e) {
                if constexpr (kWide)
                    kr[e] = *reinterpret_cast<const uint2 *>(rk + (size_t)t * DK + 4 * (s + 8 * e));
                else
                    kr[e] = *reinterpret_cast<const float4 *>(sk + (size_t)t * DK + 4 * (s + 8 * e));
            }
        };
        auto kwiden = [](KRaw r) -> float4 {
            if constexpr (kWide)
                return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                                   __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
            else
                return r;
        };
        KRaw kn[NV];
        kload(mmax - 1 < mj ? mmax - 1 : 0, kn);
        for (int t = mmax - 1; t >= 0; --t) {
            const bool live = t < mj;
            float4 k4[NV];
#pragma unroll
            for (int e = 0; e < NV; ++e) k4[e] = kwiden(kn[e]);
            if (t > 0) kload(t - 1 < mj ? t - 1 : 0, kn);
            float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < NV; ++e) acc2 = dot4x2(k4[e], u[e], acc2);
            const float d = red8(acc2.x + acc2.y);
            if (live) {
                const float bd = be[t] * d, at = al[t];
                if (s == 0) csj[t] = bd;
#pragma unroll
                for (int e = 0; e < NV; ++e) u[e] = add_ck4(scale4(at, u[e]), -at * bd, k4[e]);
            }
        }
        if (act && a.uq_nm == 0) {
            float *uqj = a.uq + (((size_t)i * a.H + h0 + hl) * a.t1max + j) * DK;
#pragma unroll
            for (int e = 0; e < NV; ++e) *reinterpret_cast<float4 *>(uqj + 4 * (s + 8 * e)) = u[e];
        } else if (act) {  // the tensor-core operand: columns 4 (s + 8 e) .. + 3 are block e, chunk s
            float *ub = a.uq + ((size_t)i * a.H + h0 + hl) * a.uq_rows * DK;
#pragma unroll
            for (int e = 0; e < NV; ++e)
                *reinterpret_cast<float4 *>(ub + ((size_t)e * a.uq_nm + j) * 32 + ((s ^ (j & 7)) << 2)) = u[e];
        }
    }
    __syncthreads();  // the weights
    // the log terms lt_j[p] = sum_{t < K + j + 1} w_j[t] v_t[p] from the staged values; a thread takes
    // four columns of a pair of step tokens (j0, j0 + 1) of one value head, so that one staged load serves
    // eight products (j0's weight past its sweep is the zero written above)
    const int nq = a.dv >> 2, npair = (T1 + 1) >> 1;
    for (int e = tid; e < hpg * npair * nq; e += nthr) {
        const int hl = e / (npair * nq), r2 = e - hl * (npair * nq), jp = r2 / nq, c = r2 - jp * nq;
        const int j0 = 2 * jp, j1 = min(j0 + 1, T1 - 1);
        const float *w0 = scw + ((size_t)hl * a.t1max + j0) * a.wcap;
        const float *w1 = scw + ((size_t)hl * a.t1max + j1) * a.wcap;
        float2 lo0 = make_float2(0.f, 0.f), hi0 = lo0, lo1 = lo0, hi1 = lo0;
        const TI *vc = svr + (size_t)hl * a.dv + 4 * c;
#pragma unroll 4
        for (int t = 0; t < K + j1 + 1; ++t) {
            const float4 v4 = lds4(vc + (size_t)t * hdv);
            const float x0 = w0[t], x1 = w1[t];
            lo0 = ffma2(make_float2(x0, x0), make_float2(v4.x, v4.y), lo0);
            hi0 = ffma2(make_float2(x0, x0), make_float2(v4.z, v4.w), hi0);
            lo1 = ffma2(make_float2(x1, x1), make_float2(v4.x, v4.y), lo1);
            hi1 = ffma2(make_float2(x1, x1), make_float2(v4.z, v4.w), hi1);
        }
        const size_t lo = (((size_t)i * a.H + h0 + hl) * a.t1max + j0) * a.dv + 4 * c;
        if (a.uq_nm) {  // the tensor-core stream, whose outputs are bf16, takes the log terms in bf16
            __nv_bfloat16 *lt0 = reinterpret_cast<__nv_bfloat16 *>(a.lt) + lo;
            *reinterpret_cast<uint2 *>(lt0) = make_uint2(bf2_pack(lo0.x, lo0.y), bf2_pack(hi0.x, hi0.y));
            if (j1 != j0)
                *reinterpret_cast<uint2 *>(lt0 + a.dv) = make_uint2(bf2_pack(lo1.x, lo1.y), bf2_pack(hi1.x, hi1.y));
        } else {
            float *lt0 = a.lt + lo;
            *reinterpret_cast<float4 *>(lt0) = make_float4(lo0.x, lo0.y, hi0.x, hi0.y);
            if (j1 != j0) *reinterpret_cast<float4 *>(lt0 + a.dv) = make_float4(lo1.x, lo1.y, hi1.x, hi1.y);
        }
    }
}

__host__ __device__ inline size_t gdn_stream_smem(int DK, int dv, int t1max) {
    return ((size_t)t1max * DK + (size_t)t1max * dv) * sizeof(float);
}

// Grid (H, batch): every checkpoint row is read once and gives the row's output for each step token:
// o_j[p] = S[p] . u_j + lt_j[p], the log term lt_j[p] = sum_{t < K + j + 1} c_j[t] v_t[p] coming from
// the coefficient kernel.
template <int DK, typename TI>
__global__ void __launch_bounds__(kGdnThreads, 2) gdn_stream_kernel(const __grid_constant__ GdnArgs a) {
    constexpr int NV = DK / 32;
    extern __shared__ __align__(16) float gsm[];
    const int h = blockIdx.x, i = blockIdx.y, slot = a.slots[i];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 3, s = lane & 7;
    if (a.slot_flags[slot] & kSlotPoisoned) return;  // flagged by the coefficient kernel
    const int T1 = a.n_tok;
    const float *st = a.state + ((size_t)slot * a.H + h) * a.dv * DK;
    // the warp's first rows are in flight while the coefficients are staged
    int pr[kRG];
    bool ok[kRG];
    float4 sv[kRG][NV];
    load_rows<NV>(st, DK, a.dv, 4 * warp, r, s, pr, ok, sv);
    float *suq = gsm;                        // [T1][DK]
    float *slt = suq + (size_t)a.t1max * DK; // [T1][dv]
    const float *uq = a.uq + ((size_t)i * a.H + h) * a.t1max * DK;
    const float *lt = a.lt + ((size_t)i * a.H + h) * a.t1max * a.dv;
    stage_rows(suq, uq, DK, T1, DK, tid, kGdnThreads);
    stage_rows(slt, lt, a.dv, T1, a.dv, tid, kGdnThreads);
    __syncthreads();
    TI *y = static_cast<TI *>(a.y);
    for (int p0 = 4 * warp; p0 < a.dv; p0 += 4 * kGdnWarps * kRG) {
        if (p0 != 4 * warp) load_rows<NV>(st, DK, a.dv, p0, r, s, pr, ok, sv);
        for (int j = 0; j < T1; ++j) {
            const float *uj = suq + (size_t)j * DK;
            float2 acc2[kRG];
#pragma unroll
            for (int q = 0; q < kRG; ++q) acc2[q] = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < NV; ++e) {
                const float4 u4 = *reinterpret_cast<const float4 *>(uj + 4 * (s + 8 * e));
#pragma unroll
                for (int q = 0; q < kRG; ++q) acc2[q] = dot4x2(sv[q][e], u4, acc2[q]);
            }
            float acc[kRG];
#pragma unroll
            for (int q = 0; q < kRG; ++q) acc[q] = acc2[q].x + acc2[q].y;
#pragma unroll
            for (int q = 0; q < kRG; ++q) acc[q] = red8(acc[q]);
            if (s == 0) {
#pragma unroll
                for (int q = 0; q < kRG; ++q)
                    if (ok[q])
                        y[(((size_t)i * T1 + j) * a.H + h) * a.dv + pr[q]] =
                            from_f<TI>(acc[q] + slt[(size_t)j * a.dv + pr[q]]);
            }
        }
    }
}

// ---------------------------------------------------------------------------- replay verify, tensor cores
//
// gdn_stream_tc_kernel: the streaming product o_j = S u_j + lt_j of bf16 pools with dk = dv = 128 on the
// 5th-generation tensor cores.  An item is one (request, value head): its 128 x 128 fp32 checkpoint is the
// A operand (M = 128 rows p, K = 128), read in place from four 32-column TMA boxes whose 128-byte swizzle
// is the K-major operand layout of kind::tf32; B is U, the swept queries, NM rows written in the same layout
// by the coefficient kernel.  kind::tf32 takes each fp32 operand through its top 19 bits (the low 13
// mantissa bits dropped), at most 2^-10 of each product, below the bf16 rounding of the outputs; fp32
// pools keep the CUDA-core kernel above.
// Warps: 0-3 epilogue (TMEM lane quarter w, thread = row p = 32 w + lane): o_j[p] = D[p][j] + lt_j[p];
//        4 per-item producer: U and the log terms of an item into a small ring (after the coefficient
//          kernel's completion);
//        5 checkpoint producer: 16 KiB boxes into a ring, a slot refilled once the MMAs of the item that
//          held it are done (so no per-slot release is needed);
//        6 MMA issuer (lane 0), 16 MMAs and one commit per item; TMEM owner.
constexpr int kGtProd = 4, kGtRing = 5, kGtMma = 6, kGtThreads = 7 * 32;
constexpr int kGtMaxRing = 12, kGtAux = 3, kGtDone = 4, kGtDbuf = 4;
constexpr int kGtMinTokens = 4;
constexpr uint32_t kGtCols = 128;  // kGtDbuf accumulators of up to 32 columns

struct GtLayout {
    uint32_t u, lt, hdr, aux, aux_base, bars;
};

// Per-item stage: U [4 column blocks][NM rows][32 fp32], the log terms [t1max][dv] bf16, a header (the gate).
__host__ __device__ inline GtLayout gt_layout(int NM, int t1max, int dv, int nring) {
    GtLayout L;
    L.u = 0;
    L.lt = 4u * (uint32_t)NM * 128u;
    L.hdr = L.lt + (uint32_t)t1max * (uint32_t)dv * 2u;
    L.aux = (L.hdr + 16u + 1023u) & ~1023u;
    L.aux_base = (uint32_t)nring * 16384u;
    L.bars = L.aux_base + kGtAux * L.aux;
    return L;
}

__host__ __device__ inline size_t gt_smem(const GtLayout &L) {
    return (size_t)L.bars + (kGtMaxRing + 2 * kGtAux + kGtDone + kGtDbuf) * 8 + 1024;
}

__device__ __forceinline__ bool gt_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort, uint32_t *flags) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && *abort) return false;
    }
    *abort = 1u;
    atomicOr(flags, SSM_FLAG_TIMEOUT);
    return false;
}

// The epilogue warps' barrier (named barrier 1, 128 threads) that ORs a predicate.
__device__ __forceinline__ bool gt_epi_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

template <int NM>
__global__ void __launch_bounds__(kGtThreads, 1)
    gdn_stream_tc_kernel(const __grid_constant__ GdnArgs a, const __grid_constant__ CUtensorMap tm_state, int nring) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t s_abort, s_tmem;
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int H = a.H, T1 = a.n_tok, dv = a.dv;  // dv = 128
    const int n_items = a.batch * H;
    const GtLayout L = gt_layout(NM, a.t1max, dv, nring);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *rfull = bars;                                     // checkpoint ring
    uint64_t *xfull = rfull + kGtMaxRing, *xempty = xfull + kGtAux;  // per-item ring
    uint64_t *done = xempty + kGtAux;                           // MMAs of an item finished
    uint64_t *dempty = done + kGtDone;                          // accumulators read
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nring; ++s) mbar_init(&rfull[s], 1);
        for (int s = 0; s < kGtAux; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], 4);
        }
        for (int s = 0; s < kGtDone; ++s) mbar_init(&done[s], 1);
        for (int s = 0; s < kGtDbuf; ++s) mbar_init(&dempty[s], 4);
        mbar_fence_init();
        s_abort = 0u;
    }
    if (warp == kGtMma) tc::tmem_alloc(&s_tmem, kGtCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    if (warp == kGtProd) {
        // ------------------------------------------------------------ per-item producer
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");  // U, the log terms and the flags are written
            int xlast[kGtAux];
            for (int s = 0; s < kGtAux; ++s) xlast[s] = -1;
            const uint32_t ubytes = 4u * NM * 128u, lbytes = (uint32_t)T1 * dv * 2u;
            for (int u = 0;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int i = item / H, h = item - i * H, slot = a.slots[i];
                const int xs = u % kGtAux;
                if (u >= kGtAux && !gt_wait(&xempty[xs], (uint32_t)((u / kGtAux) - 1) & 1u, &s_abort, a.flags)) break;
                unsigned char *X = smem + L.aux_base + (size_t)xs * L.aux;
                const int gate = (a.slot_flags[slot] & kSlotPoisoned) ? 1 : 0;
                *reinterpret_cast<int *>(X + L.hdr) = gate;
                if (gate) {
                    mbar_arrive(&xfull[xs]);
                } else {
                    mbar_arrive_expect_tx(&xfull[xs], ubytes + lbytes);
                    bulk_g2s(X + L.u, a.uq + ((size_t)i * H + h) * a.uq_rows * 128, ubytes, &xfull[xs]);
                    bulk_g2s(X + L.lt,
                             reinterpret_cast<const __nv_bfloat16 *>(a.lt) + ((size_t)i * H + h) * a.t1max * dv,
                             lbytes, &xfull[xs]);
                    xlast[xs] = u;
                }
            }
            for (int s = 0; s < kGtAux; ++s)  // no copy may still be landing when the CTA exits
                if (xlast[s] >= 0 && !mbar_wait(&xfull[s], (uint32_t)(xlast[s] / kGtAux) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp == kGtRing) {
        // ------------------------------------------------------------ checkpoint producer
        if (lane == 0) {
            int rlast[kGtMaxRing];
            for (int s = 0; s < kGtMaxRing; ++s) rlast[s] = -1;
            int nblk = 0;
            bool alive = true;
            for (int u = 0; alive; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int i = item / H, h = item - i * H;
                const int row0 = (a.slots[i] * H + h) * dv;
                for (int kb = 0; kb < 4; ++kb, ++nblk) {
                    const int rs = nblk % nring;
                    if (nblk >= nring) {  // the slot's last block belonged to item pu: its MMAs are done
                        const int pu = (nblk - nring) >> 2;
                        if (!gt_wait(&done[pu % kGtDone], (uint32_t)(pu / kGtDone) & 1u, &s_abort, a.flags)) {
                            alive = false;
                            break;
                        }
                    }
                    mbar_arrive_expect_tx(&rfull[rs], 16384u);
                    tma_load_2d(smem + (size_t)rs * 16384, &tm_state, kb * 32, row0, &rfull[rs]);
                    rlast[rs] = nblk;
                }
            }
            for (int s = 0; s < nring; ++s)  // no copy may still be landing when the CTA exits
                if (rlast[s] >= 0 && !mbar_wait(&rfull[s], (uint32_t)(rlast[s] / nring) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp == kGtMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_tf32_f32(128, NM);
            int last = -1;
            for (int u = 0;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int xs = u % kGtAux, db = u % kGtDbuf;
                if (!gt_wait(&xfull[xs], (uint32_t)(u / kGtAux) & 1u, &s_abort, a.flags)) break;
                if (u >= kGtDbuf && !gt_wait(&dempty[db], (uint32_t)((u / kGtDbuf) - 1) & 1u, &s_abort, a.flags))
                    break;
                const uint32_t d = tmem + (uint32_t)db * NM;
                const uint32_t ub = smem_addr(smem + L.aux_base + (size_t)xs * L.aux + L.u);
                bool ok = true;
                for (int kb = 0; kb < 4 && ok; ++kb) {
                    const int c = 4 * u + kb, rs = c % nring;
                    ok = gt_wait(&rfull[rs], (uint32_t)(c / nring) & 1u, &s_abort, a.flags);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t ab = smem_addr(smem + (size_t)rs * 16384);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // K = 8 tf32 per MMA
                        tc::mma_tf32(d, tc::smem_desc_sw128(ab + 32 * kk, 1024),
                                     tc::smem_desc_sw128(ub + (uint32_t)kb * NM * 128 + 32 * kk, 1024), idesc,
                                     (kb | kk) != 0);
                }
                tc::mma_commit(&done[u % kGtDone]);  // also when cut short: what was issued completes first
                last = u;
                if (!ok) break;
            }
            // every MMA issued has completed before TMEM is released
            if (last >= 0 && !mbar_wait(&done[last % kGtDone], (uint32_t)(last / kGtDone) & 1u))
                atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-3)
        const int p = 32 * warp + lane;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(a.y);
        for (int u = 0;; ++u) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            const int xs = u % kGtAux, db = u % kGtDbuf;
            const bool ok = gt_wait(&xfull[xs], (uint32_t)(u / kGtAux) & 1u, &s_abort, a.flags);
            if (gt_epi_or(!ok)) break;
            const unsigned char *X = smem + L.aux_base + (size_t)xs * L.aux;
            const int gate = *reinterpret_cast<const int *>(X + L.hdr);
            const int i = item / H, h = item - i * H;
            const bool okd = gt_wait(&done[u % kGtDone], (uint32_t)(u / kGtDone) & 1u, &s_abort, a.flags);
            if (gt_epi_or(!okd)) break;
            tc::fence_after_sync();
            float d[NM];
#pragma unroll
            for (int c = 0; c < NM; c += 16) {
                float part[16];
                tc::tmem_ld16(tmem + lane_off + (uint32_t)db * NM + c, part);
#pragma unroll
                for (int q = 0; q < 16; ++q) d[c + q] = part[q];
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[db]);
            if (!gate) {
                const __nv_bfloat16 *lt = reinterpret_cast<const __nv_bfloat16 *>(X + L.lt);
                __nv_bfloat16 *yr = y + ((size_t)i * T1 * H + h) * dv + p;
#pragma unroll
                for (int j = 0; j < NM; ++j)
                    if (j < T1)
                        yr[(size_t)j * H * dv] = __float2bfloat16_rn(d[j] + __bfloat162float(lt[(size_t)j * dv + p]));
            }
            __syncwarp();  // the stage is read (U by the MMAs, done above; the log terms here)
            if (lane == 0) mbar_arrive(&xempty[xs]);
        }
    }
    __syncwarp();  // warps whose lane 0 ran a role alone arrive at the block barrier converged
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kGtMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kGtCols);
    }
}

// ---------------------------------------------------------------------------- commit and fold

// One CTA: per request, append the kept tokens to the log or mark the request for a fold (and list it).
__global__ void gdn_commit_kernel(const __grid_constant__ GdnArgs a) {
    // the fold may be scheduled now: it waits for this grid before it reads the list
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) a.fold_list[kGdnListCount] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < a.batch; i += blockDim.x) {
        const int slot = a.slots[i];
        a.fold_m[i] = 0;
        if (a.slot_flags[slot] & kSlotPoisoned) {
            atomicOr(a.flags, SSM_FLAG_POISONED_SLOT);
            continue;
        }
        const int acc = a.accept[i];
        if (acc < 0 || acc > a.ntok[i] - 1) {
            poison(a, slot, SSM_FLAG_BAD_ACCEPT);
            continue;
        }
        const int c = acc + 1, K = a.log_len[slot];
        a.position[slot] += c;
        if (K + c < a.W && !a.force_fold) {
            a.log_len[slot] = K + c;
        } else {
            a.fold_m[i] = K + c;
            a.log_len[slot] = 0;
            reinterpret_cast<int4 *>(a.fold_list)[atomicAdd(&a.fold_list[kGdnListCount], 1)] = make_int4(i, slot, K + c, 0);
        }
    }
}

__host__ __device__ inline size_t gdn_fold_smem(int DK, int dv, int wcap) {
    return ((size_t)wcap * DK + (size_t)wcap * dv + 2 * (size_t)wcap) * sizeof(float);
}

// Grid (H, batch): the requests marked by the commit apply their M logged tokens to the checkpoint,
// row by row, in order.
template <int DK, typename TI>
__global__ void __launch_bounds__(kGdnThreads, 2) gdn_fold_kernel(const __grid_constant__ GdnArgs a) {
    constexpr int NV = DK / 32;
    extern __shared__ __align__(16) float gsm[];
    const int h = blockIdx.x, i = blockIdx.y;
    const int M = a.fold_m[i];
    if (M == 0) return;
    const int slot = a.slots[i], kh = h / a.hpg;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 3, s = lane & 7;
    float *st = a.state + ((size_t)slot * a.H + h) * a.dv * DK;
    // the warp's first rows are in flight while the logged tokens are staged
    int pr[kRG];
    bool ok[kRG];
    float4 sv[kRG][NV];
    load_rows<NV>(st, DK, a.dv, 4 * warp, r, s, pr, ok, sv);
    float *sk = gsm;                          // [M][DK]
    float *svv = sk + (size_t)a.wcap * DK;    // [M][dv]
    float *sal = svv + (size_t)a.wcap * a.dv; // [M]
    float *sbe = sal + a.wcap;                // [M]
    const TI *lk = static_cast<const TI *>(a.log_k) + (size_t)slot * a.wcap * a.G * DK;
    const TI *lv = static_cast<const TI *>(a.log_v) + (size_t)slot * a.wcap * a.H * a.dv;
    stage_rows(sk, lk + (size_t)kh * DK, (size_t)a.G * DK, M, DK, tid, kGdnThreads);
    stage_rows(svv, lv + (size_t)h * a.dv, (size_t)a.H * a.dv, M, a.dv, tid, kGdnThreads);
    for (int t = tid; t < M; t += kGdnThreads) {
        sal[t] = expf(a.log_g[((size_t)slot * a.wcap + t) * a.H + h]);
        sbe[t] = a.log_b[((size_t)slot * a.wcap + t) * a.H + h];
    }
    __syncthreads();
    for (int p0 = 4 * warp; p0 < a.dv; p0 += 4 * kGdnWarps * kRG) {
        if (p0 != 4 * warp) load_rows<NV>(st, DK, a.dv, p0, r, s, pr, ok, sv);
        // The rows are kept as sigma R with one scale for the whole head (the gate is per head), so
        // that a token costs one multiply-add per element for S . k and one for the update:
        //   w = sigma R . k,  sigma <- exp(g) sigma,  R <- R + ((beta v - exp(g) beta w) / sigma) k
        // (the same S_t = exp(g) S (I - beta k k^T) + beta v k^T); R is rescaled whenever sigma leaves
        // [2^-60, 1] or a gate is near zero.
        float sig = 1.f;
        for (int t = 0; t < M; ++t) {
            const float *kt = sk + (size_t)t * DK;
            float4 kr[NV];
#pragma unroll
            for (int e = 0; e < NV; ++e) kr[e] = *reinterpret_cast<const float4 *>(kt + 4 * (s + 8 * e));
            float w[kRG];
#pragma unroll
            for (int q = 0; q < kRG; ++q) {
                float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < NV; ++e) acc2 = dot4x2(sv[q][e], kr[e], acc2);
                w[q] = acc2.x + acc2.y;
            }
#pragma unroll
            for (int q = 0; q < kRG; ++q) w[q] = red8(w[q]) * sig;
            const float al = sal[t], be = sbe[t];
            if (al < 0x1p-20f || sig * al < 0x1p-60f) {
                // a gate near zero, or a scale about to leave fp32's range: fold the scale into the rows
                // and take this token's update directly (uniform over the CTA: both are the head's)
#pragma unroll
                for (int q = 0; q < kRG; ++q) {
                    const float c = be * svv[(size_t)t * a.dv + (ok[q] ? pr[q] : 0)] - al * be * w[q];
#pragma unroll
                    for (int e = 0; e < NV; ++e) sv[q][e] = axpy4(al * sig, sv[q][e], c, kr[e]);
                }
                sig = 1.f;
            } else {
                sig *= al;
                const float inv = 1.f / sig;
#pragma unroll
                for (int q = 0; q < kRG; ++q) {
                    const float c = (be * svv[(size_t)t * a.dv + (ok[q] ? pr[q] : 0)] - al * be * w[q]) * inv;
#pragma unroll
                    for (int e = 0; e < NV; ++e) sv[q][e] = add_ck4(sv[q][e], c, kr[e]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kRG; ++q)
#pragma unroll
            for (int e = 0; e < NV; ++e) sv[q][e] = scale4(sig, sv[q][e]);
        store_rows<NV>(st, DK, pr, ok, s, sv);
    }
}

// ---------------------------------------------------------------------------- fold, tensor cores
//
// gdn_fold_tc_kernel: the fold of bf16 pools with dk = dv = 128 and logs of at most 32 tokens, in the
// chunked (WY) form of the delta rule instead of token after token.  With G_t = g_0 + ... + g_t, unrolling
// S_t = e^{g_t} S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T from the checkpoint S gives
//   S_t = e^{G_t} S + sum_{s <= t} e^{G_t - G_s} u_s k_s^T,   u_t = b_t v_t - b_t e^{g_t} S_{t-1} k_t,
// and substituting S_{t-1} into u_t gives U (I + A) = Y over the M logged tokens, where
//   Y[p][t] = b_t v_t[p] - b_t e^{G_t} (S k_t)[p],   A[s][t] = b_t e^{G_t - G_s} (k_s . k_t) for s < t, else 0,
// so that
//   S_M = e^{G_{M-1}} S + Y P,   P = (I + A)^{-1} D K,   D = diag(e^{G_{M-1} - G_s}),
// K the M x dk keys.  I + A is unit upper triangular: P[s] = D_s k_s - sum_{t > s} A[s][t] P[t], from the
// last token back.  The products run on the tensor cores (kind::tf32): the keys' Gram matrix K K^T (the
// keys widened into the operand layout serve as both operands; A spans 128 rows, of which the 32 read
// back are the keys), X = S K^T with the checkpoint boxes read in place as A (N = 32), then Y P with Y as
// A (written over the keys once X is out) and P^T as B (K = the tokens, 8 an MMA).  e^{G_{M-1}} S is
// added in fp32 by the epilogue, so only the update passes through tf32 (2^-10 of each product, as in
// the verify's product); fp32 pools and longer logs keep the CUDA-core fold above.
//
// An item is one (folding request, value head) of the commit's list; a CTA an SM takes items in turn.
// Warps: 0-3 epilogue (thread = row p, TMEM lane quarter w): Y from X; then S_M = e^{G_{M-1}} S + Y P in
//          place in the staged boxes;
//        4-7 coefficients, into a two-stage ring: the gates' running sums (base 2), the keys widened into
//          the operand layout, the values; A from the Gram matrix (read back by warp 4 from TMEM lanes
//          0-31) and P^T.  The next item's loads are issued while an item is worked on;
//        8 checkpoint producer (lane 0): an item's four 32-column boxes into a two-stage ring; it stores
//          each item's new rows back by TMA once the epilogue has written them, and refills the stage
//          once the store has read it;
//        9 MMA issuer (lane 0) and TMEM owner: the Gram matrix as soon as the keys are in, into columns
//          256 b + 160 .. + 191; X into 256 b; Y P into 256 b + 32 .. + 159 (b = item % 2).
constexpr int kGfCoef = 4, kGfProd = 8, kGfMma = 9, kGfThreads = 10 * 32;
constexpr int kGfMaxTok = 32;
constexpr uint32_t kGfCols = 512;
constexpr uint32_t kGfState = 65536;  // four 16 KiB boxes: 128 rows x 32 fp32 each

// Per-item stage: keys [4 blocks][32 rows][32 fp32] in the B layout of S K^T (then Y [128 rows][32 fp32]),
// P^T [128 rows][32 fp32], the values [32][128] bf16 as logged, A^T [32][32], and the scalars b_t,
// b_t e^{G_t}, e^{G_{M-1} - G_t}, G_t ([4][32]) and e^{G_{M-1}}.
struct GfLayout {
    uint32_t keys, pt, vals, am, sc, aux, aux_base, bars, total;
};
__host__ __device__ constexpr GfLayout gf_layout() {
    return GfLayout{0u,
                    16384u,
                    32768u,
                    32768u + kGfMaxTok * 128u * 2u,
                    32768u + kGfMaxTok * 128u * 2u + kGfMaxTok * kGfMaxTok * 4u,
                    32768u + kGfMaxTok * 128u * 2u + kGfMaxTok * kGfMaxTok * 4u + 1024u,
                    2u * kGfState,
                    2u * kGfState + 2u * (32768u + kGfMaxTok * 128u * 2u + kGfMaxTok * kGfMaxTok * 4u + 1024u),
                    2u * kGfState + 2u * (32768u + kGfMaxTok * 128u * 2u + kGfMaxTok * kGfMaxTok * 4u + 1024u) +
                        32u * 8u + 1024u};
}

// The descriptor of an operand `bytes` past the one d was made for: the start address field (bits 0-13)
// holds the address >> 4, and shared memory addresses stay below 2^18, so the field takes the sum.
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// Named barrier id over 128 threads that ORs a predicate.
template <int ID>
__device__ __forceinline__ bool gf_bar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "n"(ID)
        : "memory");
    return r != 0;
}

// P by back substitution, right-looking: thread n holds column n, r[s] = D_s k_s[n] less the later rows'
// shares, r[t] final once every row after t is applied (the coefficient table holds -A^T); tokens from
// B on are zero (M <= B), and P^T row n goes to the B layout of Y P (chunk c: tokens 4c .. 4c + 3).
template <int B>
__device__ __forceinline__ void gf_solve(unsigned char *X, const GfLayout &L, int n, int M) {
    const float *sc = reinterpret_cast<const float *>(X + L.sc);
    const float *amt = reinterpret_cast<const float *>(X + L.am);
    const int cn = (n & 31) >> 2;
    const unsigned char *kn = X + L.keys + (n >> 5) * 4096 + (n & 3) * 4;
    float r[B];
#pragma unroll
    for (int s = 0; s < B; ++s)
        r[s] = s < M ? sc[64 + s] * *reinterpret_cast<const float *>(kn + s * 128 + ((cn ^ (s & 7)) << 4)) : 0.f;
#pragma unroll
    for (int t = B - 1; t >= 1; --t) {  // pairs of rows with the two-wide FMA
        const float2 pt = make_float2(r[t], r[t]);
#pragma unroll
        for (int s4 = 0; s4 < B; s4 += 4) {
            if (s4 < t) {
                const float4 av = *reinterpret_cast<const float4 *>(amt + t * kGfMaxTok + s4);
                if (s4 + 1 < t) {
                    const float2 v = ffma2(make_float2(av.x, av.y), pt, make_float2(r[s4], r[s4 + 1]));
                    r[s4] = v.x;
                    r[s4 + 1] = v.y;
                } else {
                    r[s4] = fmaf(av.x, pt.x, r[s4]);
                }
                if (s4 + 3 < t) {
                    const float2 v = ffma2(make_float2(av.z, av.w), pt, make_float2(r[s4 + 2], r[s4 + 3]));
                    r[s4 + 2] = v.x;
                    r[s4 + 3] = v.y;
                } else if (s4 + 2 < t) {
                    r[s4 + 2] = fmaf(av.z, pt.x, r[s4 + 2]);
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4 *>(X + L.pt + n * 128 + ((c ^ (n & 7)) << 4)) =
            4 * c < B ? make_float4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(kGfThreads, 1)
    gdn_fold_tc_kernel(const __grid_constant__ GdnArgs a, const __grid_constant__ CUtensorMap tm_state) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t s_abort, s_tmem;
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    constexpr GfLayout L = gf_layout();
    const int H = a.H, dv = 128;
    const int4 *list = reinterpret_cast<const int4 *>(a.fold_list);  // {request, slot, M, 0} per folding request
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *sfull = bars, *sready = bars + 2;  // checkpoint stages: loaded; new rows written
    uint64_t *cfull = bars + 4, *cempty = bars + 6;  // coefficient stages
    uint64_t *xdone = bars + 8, *yfull = bars + 10, *ddone = bars + 12, *tfree = bars + 14;  // TMEM buffers
    uint64_t *kfull = bars + 16;  // the keys, values and scalars of a coefficient stage (before A and P^T)
    uint64_t *gdone = bars + 18;  // the Gram matrix of a TMEM buffer
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 20; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
        s_abort = 0u;
    }
    if (warp == kGfMma) tc::tmem_alloc(&s_tmem, kGfCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    // launched programmatically after the commit kernel: the set-up above ran under it; its list is read
    // once it has completed.  The next verify's coefficient kernel may be scheduled meanwhile (it waits
    // for this grid before reading anything).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n_items = *reinterpret_cast<volatile const int32_t *>(&a.fold_list[kGdnListCount]) * H;

    if (warp == kGfProd) {
        // ------------------------------------------------------------ checkpoint producer
        // It also stores each item's new rows back (once the epilogue has written them) and reuses the stage
        // once the store has read it.
        if (lane == 0) {
            int last[2] = {-1, -1};
            auto store = [&](int v) -> bool {
                const int b = v & 1;
                if (!gt_wait(&sready[b], (uint32_t)(v >> 1) & 1u, &s_abort, a.flags)) return false;
                const int item = blockIdx.x + v * gridDim.x;
                const int f = item / H, h = item - f * H, slot = list[f].y;
                for (int kb = 0; kb < 4; ++kb)
                    tma_store_2d(&tm_state, kb * 32, (slot * H + h) * dv, smem + (size_t)b * kGfState + kb * 16384);
                bulk_commit();
                bulk_wait_read0();
                return true;
            };
            int u = 0;
            bool ok = true;
            for (;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int f = item / H, h = item - f * H, slot = list[f].y;
                const int b = u & 1;
                if (u >= 2 && !(ok = store(u - 2))) break;
                mbar_arrive_expect_tx(&sfull[b], kGfState);
                for (int kb = 0; kb < 4; ++kb)
                    tma_load_2d(smem + (size_t)b * kGfState + kb * 16384, &tm_state, kb * 32, (slot * H + h) * dv,
                                &sfull[b]);
                last[b] = u;
            }
            for (int v = u >= 2 ? u - 2 : 0; ok && v < u; ++v) ok = store(v);
            bulk_wait0();  // every store has landed before the CTA exits
            for (int b = 0; b < 2; ++b)  // and no load is still landing
                if (last[b] >= 0 && !mbar_wait(&sfull[b], (uint32_t)(last[b] >> 1) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp >= kGfCoef && warp < kGfCoef + 4) {
        // ------------------------------------------------------------ coefficients
        // An item's loads are issued while the item before it is worked on: its values by async copies into
        // its stage (once the stage is free), its keys (eight 4-value pieces a thread: token t = ct / 32 + 4 j,
        // column 4 (ct % 32)) and gates (warp 4, a lane a token) into registers.
        const int ct = threadIdx.x - 32 * kGfCoef, c4 = ct & 31;
        uint2 kraw[8];
        float gn = 0.f, bn = 0.f;
        int mn = 0;
        // the list entry of the item the next issue() takes, loaded one call ahead
        auto entry = [&](int u) -> int4 {
            const int item = blockIdx.x + u * gridDim.x;
            return item < n_items ? list[item / H] : make_int4(0, 0, 0, 0);
        };
        int4 fq = entry(0);
        auto issue = [&](int u) -> bool {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) return true;
            const int4 fe = fq;
            const int h = item - (item / H) * H, slot = fe.y, kh = h / a.hpg;
            const int M = fe.z, b = u & 1;
            mn = M;
            const bool ok = u < 2 || gt_wait(&cempty[b], (uint32_t)((u >> 1) - 1) & 1u, &s_abort, a.flags);
            if (gf_bar_or<2>(!ok)) return false;
            unsigned char *X = smem + L.aux_base + (size_t)b * L.aux;
            const __nv_bfloat16 *lv =
                static_cast<const __nv_bfloat16 *>(a.log_v) + ((size_t)slot * a.wcap * H + h) * dv;
            for (int e = ct; e < M * 16; e += 128) {  // 16-byte pieces of the M value rows
                const int t = e >> 4, c = e & 15;
                cp_async16(X + L.vals + t * 256 + c * 16, lv + (size_t)t * H * dv + c * 8);
            }
            cp_async_commit();
            const __nv_bfloat16 *lk =
                static_cast<const __nv_bfloat16 *>(a.log_k) + ((size_t)slot * a.wcap * a.G + kh) * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = (ct >> 5) + 4 * j;
                kraw[j] = t < M ? *reinterpret_cast<const uint2 *>(lk + (size_t)t * a.G * 128 + 4 * c4) : make_uint2(0u, 0u);
            }
            if (ct < 32) {
                const size_t o = ((size_t)slot * a.wcap + ct) * H + h;
                gn = ct < M ? a.log_g[o] : 0.f;
                bn = ct < M ? a.log_b[o] : 0.f;
            }
            fq = entry(u + 1);
            return true;
        };
        bool alive = issue(0);
        for (int u = 0; alive; ++u) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            const int M = mn;
            const int b = u & 1;
            unsigned char *X = smem + L.aux_base + (size_t)b * L.aux;
            float *sc = reinterpret_cast<float *>(X + L.sc);
            float *amt = reinterpret_cast<float *>(X + L.am);  // A^T [t][s]
            if (ct < 32) {  // the gates' running sums, a lane a token (zero past M)
                const int t = ct;
                float G = gn;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, G, off);
                    if (t >= off) G += n;
                }
                G *= 1.4426950408889634f;  // base 2 from here on
                const float GM = __shfl_sync(0xffffffffu, G, M - 1);
                sc[t] = bn;
                sc[32 + t] = t < M ? bn * exp2f(G) : 0.f;
                sc[64 + t] = t < M ? exp2f(GM - G) : 0.f;
                sc[96 + t] = G;
                if (t == 0) sc[128] = exp2f(GM);
            }
            // the keys widened into the operand layout (block n / 32, row t, 16-byte chunk ((n % 32) / 4) ^ (t % 8))
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = (ct >> 5) + 4 * j;
                const uint2 r = kraw[j];
                *reinterpret_cast<float4 *>(X + L.keys + (c4 >> 3) * 4096 + t * 128 + (((c4 & 7) ^ (t & 7)) << 4)) =
                    make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u),
                                __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xFFFF0000u));
            }
            cp_async_wait<0>();            // this item's values
            tc::fence_proxy_async_smem();  // the keys are read by the tensor cores
            bar_sync_named(2, 128);
            if (ct == 0) mbar_arrive(&kfull[b]);  // the MMA warp starts the Gram matrix at once
            if (!issue(u + 1)) break;  // the next item's loads land during this one's work
            {  // -A^T[t][s] (zero unless s < t < M) from the Gram matrix: warp 4's lane s copies row s out of
               // TMEM into the P^T region (rows 33 floats apart, so that the copy and the reads below take
               // every bank once), then thread (t, q) forms the entries s = 8q .. 8q + 7 of row t
                float *graw = reinterpret_cast<float *>(X + L.pt);
                bool okg = true;
                if (ct < 32) {
                    okg = gt_wait(&gdone[b], (uint32_t)(u >> 1) & 1u, &s_abort, a.flags);
                    if (__all_sync(0xffffffffu, okg)) {
                        tc::fence_after_sync();
                        float gr[32];
                        tc::tmem_ld32(tmem + 256u * (uint32_t)b + 160u, gr);
#pragma unroll
                        for (int t = 0; t < kGfMaxTok; ++t) graw[ct * 33 + t] = gr[t];
                        tc::fence_before_sync();
                    } else {
                        okg = false;
                    }
                }
                if (gf_bar_or<2>(!okg)) break;
                const int t = ct >> 2, s0 = (ct & 3) * 8;
                const float nbt = -sc[t], Gt = sc[96 + t];
                float av[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (t < M)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (s0 + j < t) av[j] = nbt * exp2f(Gt - sc[96 + s0 + j]) * graw[(s0 + j) * 33 + t];
                *reinterpret_cast<float4 *>(amt + t * kGfMaxTok + s0) = make_float4(av[0], av[1], av[2], av[3]);
                *reinterpret_cast<float4 *>(amt + t * kGfMaxTok + s0 + 4) = make_float4(av[4], av[5], av[6], av[7]);
                bar_sync_named(2, 128);
            }
            // P by back substitution (rows past M come out zero), at the item's token bound
            switch ((M + 7) >> 3) {
            case 1: gf_solve<8>(X, L, ct, M); break;
            case 2: gf_solve<16>(X, L, ct, M); break;
            case 3: gf_solve<24>(X, L, ct, M); break;
            default: gf_solve<32>(X, L, ct, M); break;
            }
            tc::fence_proxy_async_smem();  // P^T is read by the tensor cores
            bar_sync_named(2, 128);
            if (ct == 0) mbar_arrive(&cfull[b]);
        }
        cp_async_wait<0>();  // no copy may still be landing when the CTA exits
    } else if (warp == kGfMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idx = tc::idesc_tf32_f32(128, 32), idd = tc::idesc_tf32_f32(128, 128);
            uint64_t *lastb = nullptr;
            uint32_t lastph = 0;
            for (int u = 0;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int M = list[item / H].z;
                const int b = u & 1;
                const uint32_t ph = (uint32_t)(u >> 1) & 1u;
                if (u >= 2 && !gt_wait(&tfree[b], ph ^ 1u, &s_abort, a.flags)) break;
                if (!gt_wait(&kfull[b], ph, &s_abort, a.flags)) break;
                tc::fence_after_sync();
                const uint32_t sb = smem_addr(smem + (size_t)b * kGfState);
                const uint32_t xb = smem_addr(smem + L.aux_base + (size_t)b * L.aux);
                const uint32_t dx = tmem + 256u * (uint32_t)b, dd = dx + 32u, dg = dx + 160u;
                const uint64_t dk0 = tc::smem_desc_sw128(xb + L.keys, 1024);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)  // the Gram matrix: rows past 32 of A are not read back
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t d = desc_at(dk0, kb * 4096 + 32 * kk);
                        tc::mma_tf32(dg, d, d, idx, (kb | kk) != 0);
                    }
                tc::mma_commit(&gdone[b]);
                lastb = &gdone[b];
                lastph = ph;
                if (!gt_wait(&sfull[b], ph, &s_abort, a.flags)) break;
                tc::fence_after_sync();
                const uint64_t ds0 = tc::smem_desc_sw128(sb, 1024);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // K = 8 tf32 per MMA
                        tc::mma_tf32(dx, desc_at(ds0, kb * 16384 + 32 * kk), desc_at(dk0, kb * 4096 + 32 * kk), idx,
                                     (kb | kk) != 0);
                tc::mma_commit(&xdone[b]);
                lastb = &xdone[b];
                lastph = ph;
                if (!gt_wait(&cfull[b], ph, &s_abort, a.flags)) break;
                if (!gt_wait(&yfull[b], ph, &s_abort, a.flags)) break;
                tc::fence_after_sync();
                const uint64_t dp0 = tc::smem_desc_sw128(xb + L.pt, 1024);
                for (int kk = 0; kk < (M + 7) / 8; ++kk)
                    tc::mma_tf32(dd, desc_at(dk0, 32 * kk), desc_at(dp0, 32 * kk), idd, kk != 0);
                tc::mma_commit(&ddone[b]);
                lastb = &ddone[b];
            }
            // every MMA issued has completed before TMEM is released
            if (lastb && !mbar_wait(lastb, lastph)) atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        const int p = threadIdx.x;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        for (int u = 0;; ++u) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            const int M = list[item / H].z;
            const int b = u & 1;
            const uint32_t ph = (uint32_t)(u >> 1) & 1u;
            unsigned char *X = smem + L.aux_base + (size_t)b * L.aux;
            unsigned char *S = smem + (size_t)b * kGfState;
            bool ok = gt_wait(&kfull[b], ph, &s_abort, a.flags) && gt_wait(&sfull[b], ph, &s_abort, a.flags) &&
                      gt_wait(&xdone[b], ph, &s_abort, a.flags);
            if (gf_bar_or<1>(!ok)) break;
            tc::fence_after_sync();
            float x[32];
            tc::tmem_ld32(tmem + lane_off + 256u * (uint32_t)b, x);
            const float *sc = reinterpret_cast<const float *>(X + L.sc);
            const __nv_bfloat16 *vals = reinterpret_cast<const __nv_bfloat16 *>(X + L.vals);
            const float gam = sc[128];
#pragma unroll
            for (int t = 0; t < 32; ++t)
                x[t] = t < M ? fmaf(sc[t], __bfloat162float(vals[t * 128 + p]), -sc[32 + t] * x[t]) : 0.f;
            // Y row p over the keys, once the coefficient warps are done with them (and X is out): chunk c
            // holds tokens 4c .. 4c + 3
            ok = gt_wait(&cfull[b], ph, &s_abort, a.flags);
            if (gf_bar_or<1>(!ok)) break;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4 *>(X + L.keys + p * 128 + ((c ^ (p & 7)) << 4)) =
                    make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            bar_sync_named(1, 128);
            if (p == 0) mbar_arrive(&yfull[b]);
            ok = gt_wait(&ddone[b], ph, &s_abort, a.flags);
            if (gf_bar_or<1>(!ok)) break;
            tc::fence_after_sync();
            if (p == 0) mbar_arrive(&cempty[b]);  // Y and P^T are read; the values and scalars were read above
            // S_M = e^{G_{M-1}} S + Y P, row p, in place in the staged boxes
#pragma unroll 1
            for (int kb = 0; kb < 4; ++kb) {
                float d[32];
                tc::tmem_ld32(tmem + lane_off + 256u * (uint32_t)b + 32u + 32u * (uint32_t)kb, d);
                unsigned char *row = S + kb * 16384 + p * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float4 *q = reinterpret_cast<float4 *>(row + ((c ^ (p & 7)) << 4));
                    float4 s4 = *q;
                    s4.x = fmaf(gam, s4.x, d[4 * c]);
                    s4.y = fmaf(gam, s4.y, d[4 * c + 1]);
                    s4.z = fmaf(gam, s4.z, d[4 * c + 2]);
                    s4.w = fmaf(gam, s4.w, d[4 * c + 3]);
                    *q = s4;
                }
            }
            tc::fence_before_sync();
            tc::fence_proxy_async_smem();  // the new rows are read by the producer's TMA store
            bar_sync_named(1, 128);
            if (p == 0) {
                mbar_arrive(&tfree[b]);
                mbar_arrive(&sready[b]);
            }
        }
    }
    __syncwarp();  // warps whose lane 0 ran a role alone arrive at the block barrier converged
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kGfMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kGfCols);
    }
}

// ---------------------------------------------------------------------------- reset and gather

__global__ void gdn_reset_kernel(const __grid_constant__ GdnArgs a, size_t per_slot) {
    const int slot = a.slots[blockIdx.y];
    float4 *st = reinterpret_cast<float4 *>(a.state + (size_t)slot * per_slot);
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < per_slot / 4; e += (size_t)gridDim.x * blockDim.x)
        st[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        a.log_len[slot] = 0;
        a.position[slot] = 0;
        a.slot_flags[slot] = 0u;
    }
}

__global__ void gdn_gather_kernel(const __grid_constant__ GdnArgs a, size_t per_slot, float *dst) {
    const int slot = a.slots[blockIdx.y];
    const float4 *src = reinterpret_cast<const float4 *>(a.state + (size_t)slot * per_slot);
    float4 *d = reinterpret_cast<float4 *>(dst + (size_t)blockIdx.y * per_slot);
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < per_slot / 4; e += (size_t)gridDim.x * blockDim.x)
        d[e] = src[e];
}

}  // namespace
}  // namespace ssm

// ---------------------------------------------------------------------------- host: the pool

struct ssm_gdn_pool_s {
    ssm_gdn_config cfg{};
    int n_slots = 0, device = 0, wcap = 0, in_b = 4, scratch_rows = 0;
    size_t per_slot = 0;  // floats of one slot's state
    float *state = nullptr;
    void *log_k = nullptr, *log_v = nullptr;
    float *log_g = nullptr, *log_b = nullptr, *uq = nullptr, *lt = nullptr;
    int32_t *log_len = nullptr, *fold_m = nullptr, *fold_list = nullptr;
    int64_t *position = nullptr;
    uint32_t *slot_flags = nullptr, *flags = nullptr;
    std::vector<int> pending_ntok;  // tokens of each slot's last verify (0: none since its commit)
    // bf16 pools with dk = dv = 128: the tensor-core streaming verify (rows of 128 fp32, 32-column boxes,
    // 128-byte swizzle) and the rows of U per (request, head) in its operand layout
    CUtensorMap tm_state;
    bool tc_ok = false;
    int uq_rows = 0;
    const char *last_path = "none";
    // the tensor-core fold (the same boxes; logs of at most 32 tokens)
    bool fold_tc_ok = false;
    const char *commit_path = "none";
};

namespace ssm {
namespace {

struct GdnDevice {  // the pool's device current for the call, the caller's restored after
    int prev = -1;
    explicit GdnDevice(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    }
    ~GdnDevice() {
        int now = -1;
        if (prev >= 0 && cudaGetDevice(&now) == cudaSuccess && now != prev) cudaSetDevice(prev);
    }
};

ssm_status gdn_cuda(cudaError_t e) { return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA; }

void gdn_free(ssm_gdn_pool_s *p) {
    void *bufs[] = {p->state, p->log_k, p->log_v, p->log_g, p->log_b, p->uq, p->lt,
                    p->log_len, p->fold_m, p->fold_list, p->position, p->slot_flags, p->flags};
    for (void *b : bufs)
        if (b) cudaFree(b);
}

template <typename T>
cudaError_t gdn_alloc(T **ptr, size_t count) {
    return cudaMalloc(reinterpret_cast<void **>(ptr), std::max<size_t>(count, 1) * sizeof(T));
}

GdnArgs gdn_args(const ssm_gdn_pool_s &p) {
    GdnArgs a;
    std::memset(&a, 0, offsetof(GdnArgs, slots));
    a.state = p.state;
    a.log_k = p.log_k;
    a.log_v = p.log_v;
    a.log_g = p.log_g;
    a.log_b = p.log_b;
    a.log_len = p.log_len;
    a.position = p.position;
    a.slot_flags = p.slot_flags;
    a.flags = p.flags;
    a.uq = p.uq;
    a.lt = p.lt;
    a.fold_m = p.fold_m;
    a.fold_list = p.fold_list;
    a.H = p.cfg.nheads;
    a.G = p.cfg.nkheads;
    a.hpg = p.cfg.nheads / p.cfg.nkheads;
    a.dv = p.cfg.dv;
    a.W = p.cfg.window;
    a.wcap = p.wcap;
    a.t1max = p.cfg.max_tokens;
    return a;
}

// q, k, v and y are read and written four values at a time
bool gdn_aligned(const void *q, const void *k, const void *v, const void *y) {
    return ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
             reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
}

ssm_status gdn_check_slots(const ssm_gdn_pool_s *p, const int32_t *slots, int n) {
    if (!slots || n < 1) return SSM_ERR_INVALID_ARG;
    std::vector<char> seen((size_t)p->n_slots, 0);
    for (int i = 0; i < n; ++i) {
        const int s = slots[i];
        if (s < 0 || s >= p->n_slots || seen[(size_t)s]) return SSM_ERR_INVALID_ARG;
        seen[(size_t)s] = 1;
    }
    return SSM_OK;
}

template <typename Kernel>
cudaError_t gdn_smem(Kernel k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// A launch that may begin while the stream's previous kernel drains (programmatic dependent launch):
// the kernel waits for that grid (griddepcontrol.wait) before it reads anything the grid writes.
template <typename... KArgs, typename... Args>
cudaError_t gdn_launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                           Args &&...args) {
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

// dk and the input type as template arguments
#define GDN_DISPATCH(p, ...)                                                                   \
    do {                                                                                       \
        if ((p).cfg.dk == 128) {                                                               \
            constexpr int DK = 128;                                                            \
            if ((p).in_b == 2) { using TI = __nv_bfloat16; __VA_ARGS__; }                      \
            else { using TI = float; __VA_ARGS__; }                                            \
        } else {                                                                               \
            constexpr int DK = 64;                                                             \
            if ((p).in_b == 2) { using TI = __nv_bfloat16; __VA_ARGS__; }                      \
            else { using TI = float; __VA_ARGS__; }                                            \
        }                                                                                      \
    } while (0)

// Run fn(args, first request, count) over launches of at most kGdnMaxBatch requests.
template <typename Fn>
ssm_status gdn_batches(const ssm_gdn_pool_s &p, const int32_t *slots, int batch, Fn fn) {
    GdnArgs a = gdn_args(p);
    for (int base = 0; base < batch; base += kGdnMaxBatch) {
        const int m = std::min(batch - base, kGdnMaxBatch);
        a.batch = m;
        for (int i = 0; i < m; ++i) a.slots[i] = slots[base + i];
        const cudaError_t e = fn(a, base, m);
        if (e != cudaSuccess) return gdn_cuda(e);
    }
    return SSM_OK;
}

}  // namespace
}  // namespace ssm

using ssm::GdnArgs;

extern "C" {

ssm_status ssm_gdn_init(const ssm_gdn_config *cfg, int32_t n_slots, const float *init_state, ssm_stream_t stream,
                        ssm_gdn_pool *out) {
    if (!cfg || !out || n_slots < 1) return SSM_ERR_INVALID_ARG;
    const ssm_gdn_config c = *cfg;
    if (c.nheads < 1 || c.nkheads < 1 || c.nheads % c.nkheads || (c.dk != 64 && c.dk != 128) || c.dv < 4 ||
        c.dv > 256 || c.dv % 4 || (c.input_dtype != SSM_DTYPE_F32 && c.input_dtype != SSM_DTYPE_BF16) ||
        c.window < 1 || c.window > ssm::kGdnMaxWindow || c.max_tokens < 1 || c.max_tokens > ssm::kGdnMaxTokens)
        return SSM_ERR_INVALID_ARG;
    {  // the verify and fold kernels' shared-memory working sets must fit one CTA
        int dev = 0, max_smem = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            max_smem = 0;
        const int wcap = c.window - 1 + c.max_tokens, hpg = c.nheads / c.nkheads;
        const size_t need = std::max({ssm::gdn_coef_smem(c.dk, c.dv, wcap, c.max_tokens, hpg,
                                                         c.input_dtype == SSM_DTYPE_BF16 ? 2 : 4),
                                      ssm::gdn_stream_smem(c.dk, c.dv, c.max_tokens),
                                      ssm::gdn_fold_smem(c.dk, c.dv, wcap)});
        if (max_smem > 0 && need + 1024 > (size_t)max_smem) return SSM_ERR_INVALID_ARG;
    }
    auto *p = new (std::nothrow) ssm_gdn_pool_s();
    if (!p) return SSM_ERR_NO_MEMORY;
    p->cfg = c;
    p->n_slots = n_slots;
    p->wcap = c.window - 1 + c.max_tokens;
    p->in_b = c.input_dtype == SSM_DTYPE_BF16 ? 2 : 4;
    p->per_slot = (size_t)c.nheads * c.dv * c.dk;
    p->scratch_rows = std::min(n_slots, ssm::kGdnMaxBatch);
    p->pending_ntok.assign((size_t)n_slots, 0);
    cudaGetDevice(&p->device);
    const size_t ns = (size_t)n_slots, H = (size_t)c.nheads, G = (size_t)c.nkheads, W = (size_t)p->wcap;
    const size_t sr = (size_t)p->scratch_rows, T = (size_t)c.max_tokens;
    cudaError_t e = ssm::gdn_alloc(&p->state, ns * p->per_slot);
    if (e == cudaSuccess) e = cudaMalloc(&p->log_k, ns * W * G * c.dk * p->in_b);
    if (e == cudaSuccess) e = cudaMalloc(&p->log_v, ns * W * H * c.dv * p->in_b);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->log_g, ns * W * H);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->log_b, ns * W * H);
    const bool tc_shape = p->in_b == 2 && c.dk == 128 && c.dv == 128 && c.max_tokens <= 32;
    p->uq_rows = tc_shape ? (c.max_tokens <= 16 ? 16 : 32) : c.max_tokens;
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->uq, sr * H * (size_t)p->uq_rows * c.dk);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->lt, sr * H * T * (size_t)c.dv);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->log_len, ns);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->fold_m, (size_t)ssm::kGdnMaxBatch);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->fold_list, (size_t)ssm::kGdnListCount + 1);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->position, ns);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->slot_flags, ns);
    if (e == cudaSuccess) e = ssm::gdn_alloc(&p->flags, 1);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (e == cudaSuccess) {
        e = init_state ? cudaMemcpyAsync(p->state, init_state, ns * p->per_slot * sizeof(float),
                                         cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(p->state, 0, ns * p->per_slot * sizeof(float), s);
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(p->log_len, 0, ns * sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->fold_m, 0, ssm::kGdnMaxBatch * sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->position, 0, ns * sizeof(int64_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->slot_flags, 0, ns * sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->flags, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        ssm::gdn_free(p);
        delete p;
        return e == cudaErrorMemoryAllocation ? SSM_ERR_NO_MEMORY : SSM_ERR_CUDA;
    }
    if (tc_shape) {  // else (or with no encoder in the driver) the CUDA-core streaming kernel serves
        const ssm::TensorMapEncode enc = ssm::tensor_map_encoder();
        const cuuint64_t dims[2] = {(cuuint64_t)c.dk, (cuuint64_t)ns * H * c.dv};
        const cuuint64_t strides[1] = {(cuuint64_t)c.dk * 4};
        const cuuint32_t box[2] = {32u, 128u}, es[2] = {1u, 1u};
        p->tc_ok = enc && enc(&p->tm_state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p->state, dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        int max_smem = 0;
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
        p->fold_tc_ok = p->tc_ok && p->wcap <= ssm::kGfMaxTok && ssm::gf_layout().total <= (uint32_t)max_smem;
    }
    *out = p;
    return SSM_OK;
}

ssm_status ssm_gdn_destroy(ssm_gdn_pool pool) {
    if (!pool) return SSM_ERR_INVALID_ARG;
    ssm::GdnDevice g(pool->device);
    cudaDeviceSynchronize();
    ssm::gdn_free(pool);
    delete pool;
    return SSM_OK;
}

ssm_status ssm_gdn_reset(ssm_gdn_pool pool, const int32_t *slots, int32_t n, ssm_stream_t stream) {
    if (!pool) return SSM_ERR_INVALID_ARG;
    ssm_status st = ssm::gdn_check_slots(pool, slots, n);
    if (st != SSM_OK) return st;
    ssm::GdnDevice g(pool->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t per_slot = pool->per_slot;
    st = ssm::gdn_batches(*pool, slots, n, [&](const GdnArgs &a, int, int m) {
        ssm::gdn_reset_kernel<<<dim3(16, m), 256, 0, s>>>(a, per_slot);
        return cudaGetLastError();
    });
    if (st == SSM_OK)
        for (int i = 0; i < n; ++i) pool->pending_ntok[(size_t)slots[i]] = 0;
    return st;
}

ssm_status ssm_gdn_gather(ssm_gdn_pool pool, int32_t n, const int32_t *slots, float *dst, ssm_stream_t stream) {
    if (!pool || !dst) return SSM_ERR_INVALID_ARG;
    ssm_status st = ssm::gdn_check_slots(pool, slots, n);
    if (st != SSM_OK) return st;
    ssm::GdnDevice g(pool->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t per_slot = pool->per_slot;
    return ssm::gdn_batches(*pool, slots, n, [&](const GdnArgs &a, int base, int m) {
        ssm::gdn_gather_kernel<<<dim3(16, m), 256, 0, s>>>(a, per_slot, dst + (size_t)base * per_slot);
        return cudaGetLastError();
    });
}

ssm_status ssm_gdn_decode_step(ssm_gdn_pool pool, int32_t batch, const int32_t *slots, const void *q,
                               const void *k, const void *v, const float *g, const float *beta, void *y,
                               ssm_stream_t stream) {
    if (!pool || !q || !k || !v || !g || !beta || !y || !ssm::gdn_aligned(q, k, v, y)) return SSM_ERR_INVALID_ARG;
    ssm_status st = ssm::gdn_check_slots(pool, slots, batch);
    if (st != SSM_OK) return st;
    ssm::GdnDevice dg(pool->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const ssm_gdn_pool_s &p = *pool;
    const size_t G = (size_t)p.cfg.nkheads, H = (size_t)p.cfg.nheads, dk = (size_t)p.cfg.dk, dv = (size_t)p.cfg.dv;
    const size_t ib = (size_t)p.in_b;
    st = ssm::gdn_batches(p, slots, batch, [&](GdnArgs &a, int base, int m) {
        const size_t b0 = (size_t)base;
        a.q = static_cast<const char *>(q) + b0 * G * dk * ib;
        a.k = static_cast<const char *>(k) + b0 * G * dk * ib;
        a.v = static_cast<const char *>(v) + b0 * H * dv * ib;
        a.g = g + b0 * H;
        a.beta = beta + b0 * H;
        a.y = static_cast<char *>(y) + b0 * H * dv * ib;
        cudaError_t e = cudaSuccess;
        GDN_DISPATCH(p, { ssm::gdn_decode_kernel<DK, TI><<<dim3((unsigned)H, m), ssm::kGdnThreads, 0, s>>>(a); });
        e = cudaGetLastError();
        return e;
    });
    if (st == SSM_OK)
        for (int i = 0; i < batch; ++i) pool->pending_ntok[(size_t)slots[i]] = 0;
    return st;
}

ssm_status ssm_gdn_verify_replay(ssm_gdn_pool pool, int32_t batch, int32_t n_tok, const int32_t *slots,
                                 const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 void *y, ssm_stream_t stream) {
    if (!pool || !q || !k || !v || !g || !beta || !y || !ssm::gdn_aligned(q, k, v, y)) return SSM_ERR_INVALID_ARG;
    if (n_tok < 1 || n_tok > pool->cfg.max_tokens) return SSM_ERR_INVALID_ARG;
    ssm_status st = ssm::gdn_check_slots(pool, slots, batch);
    if (st != SSM_OK) return st;
    ssm::GdnDevice dg(pool->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const ssm_gdn_pool_s &p = *pool;
    const size_t G = (size_t)p.cfg.nkheads, H = (size_t)p.cfg.nheads, dk = (size_t)p.cfg.dk, dv = (size_t)p.cfg.dv;
    const size_t ib = (size_t)p.in_b, T = (size_t)n_tok;
    const size_t csm =
        ssm::gdn_coef_smem(p.cfg.dk, p.cfg.dv, p.wcap, p.cfg.max_tokens, p.cfg.nheads / p.cfg.nkheads, p.in_b);
    // the coefficient kernel's block: four sweeps a warp; at least three warps, for the staging and the
    // log terms (few sweeps, as in a one-token step, run best at three: more CTAs an SM)
    const int nsw = (p.cfg.nheads / p.cfg.nkheads) * n_tok;
    const unsigned coef_threads = (unsigned)(32 * std::min(ssm::kGdnWarps, std::max(3, (nsw + 3) / 4)));
    const size_t ssm_ = ssm::gdn_stream_smem(p.cfg.dk, p.cfg.dv, p.cfg.max_tokens);
    // the tensor-core streaming kernel: as many 16 KiB checkpoint slots as fit beside its per-item ring
    const int NM = n_tok <= 16 ? 16 : 32;
    int nring = 0;
    size_t tsm = 0;
    // (from four step tokens: below that the CUDA-core kernel's few products per state element are cheaper
    // than the tensor-core kernel's per-item pipeline)
    if (p.tc_ok && n_tok >= ssm::kGtMinTokens && n_tok <= 32 && NM <= p.uq_rows) {
        int max_smem = 0;
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.device);
        for (int nr = ssm::kGtMaxRing; nr >= 8 && !nring; --nr) {
            const size_t b = ssm::gt_smem(ssm::gt_layout(NM, p.cfg.max_tokens, p.cfg.dv, nr));
            if (b <= (size_t)max_smem) {
                nring = nr;
                tsm = b;
            }
        }
    }
    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p.device);
    st = ssm::gdn_batches(p, slots, batch, [&](GdnArgs &a, int base, int m) {
        const size_t b0 = (size_t)base;
        a.n_tok = n_tok;
        a.uq_nm = nring ? NM : 0;
        a.uq_rows = p.uq_rows;
        a.q = static_cast<const char *>(q) + b0 * T * G * dk * ib;
        a.k = static_cast<const char *>(k) + b0 * T * G * dk * ib;
        a.v = static_cast<const char *>(v) + b0 * T * H * dv * ib;
        a.g = g + b0 * T * H;
        a.beta = beta + b0 * T * H;
        a.y = static_cast<char *>(y) + b0 * T * H * dv * ib;
        cudaError_t e = cudaSuccess;
        GDN_DISPATCH(p, {
            auto kc = ssm::gdn_coef_kernel<DK, TI>;
            auto ks = ssm::gdn_stream_kernel<DK, TI>;
            e = ssm::gdn_smem(kc, csm);
            if (e == cudaSuccess) e = ssm::gdn_smem(ks, ssm_);
            if (e == cudaSuccess) e = ssm::gdn_launch_pdl(kc, dim3((unsigned)G, m), dim3(coef_threads), csm, s, a);
            if (e == cudaSuccess) {
                if (nring) {  // bf16, dk = dv = 128: the tensor-core streaming kernel
                    auto kt = NM == 16 ? ssm::gdn_stream_tc_kernel<16> : ssm::gdn_stream_tc_kernel<32>;
                    e = ssm::gdn_smem(kt, tsm);
                    if (e == cudaSuccess)
                        e = ssm::gdn_launch_pdl(kt, dim3((unsigned)std::min<size_t>((size_t)m * H, (size_t)sms)),
                                                dim3(ssm::kGtThreads), tsm, s, a, p.tm_state, nring);
                } else {
                    ks<<<dim3((unsigned)H, m), ssm::kGdnThreads, ssm_, s>>>(a);
                }
                if (e == cudaSuccess) e = cudaGetLastError();
            }
        });
        return e;
    });
    if (st == SSM_OK) {
        for (int i = 0; i < batch; ++i) pool->pending_ntok[(size_t)slots[i]] = n_tok;
        pool->last_path = nring ? "gdn_verify_tc" : "gdn_verify";
    }
    return st;
}

ssm_status ssm_gdn_commit(ssm_gdn_pool pool, int32_t batch, const int32_t *slots, const int32_t *accept,
                          int32_t force_fold, ssm_stream_t stream) {
    if (!pool || !accept) return SSM_ERR_INVALID_ARG;
    ssm_status st = ssm::gdn_check_slots(pool, slots, batch);
    if (st != SSM_OK) return st;
    for (int i = 0; i < batch; ++i)
        if (pool->pending_ntok[(size_t)slots[i]] < 1) return SSM_ERR_INVALID_STATE;
    ssm::GdnDevice dg(pool->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const ssm_gdn_pool_s &p = *pool;
    const size_t fsm = ssm::gdn_fold_smem(p.cfg.dk, p.cfg.dv, p.wcap);
    const unsigned H = (unsigned)p.cfg.nheads;
    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p.device);
    st = ssm::gdn_batches(p, slots, batch, [&](GdnArgs &a, int base, int m) {
        a.accept = accept + base;
        a.force_fold = force_fold ? 1 : 0;
        for (int i = 0; i < m; ++i) a.ntok[i] = pool->pending_ntok[(size_t)slots[base + i]];
        ssm::gdn_commit_kernel<<<1, 1024, 0, s>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (p.fold_tc_ok) {  // persistent over the listed (request, value head) items, one CTA an SM
            const uint32_t gsm = ssm::gf_layout().total;
            e = ssm::gdn_smem(ssm::gdn_fold_tc_kernel, gsm);
            if (e != cudaSuccess) return e;
            e = ssm::gdn_launch_pdl(ssm::gdn_fold_tc_kernel, dim3((unsigned)sms), dim3(ssm::kGfThreads), gsm, s, a,
                                    p.tm_state);
            pool->commit_path = "gdn_fold_tc";
            return e;
        }
        pool->commit_path = "gdn_fold";
        GDN_DISPATCH(p, {
            auto kf = ssm::gdn_fold_kernel<DK, TI>;
            e = ssm::gdn_smem(kf, fsm);
            if (e == cudaSuccess) {
                kf<<<dim3(H, m), ssm::kGdnThreads, fsm, s>>>(a);
                e = cudaGetLastError();
            }
        });
        return e;
    });
    if (st == SSM_OK)
        for (int i = 0; i < batch; ++i) pool->pending_ntok[(size_t)slots[i]] = 0;
    return st;
}

ssm_status ssm_gdn_slot_info(ssm_gdn_pool pool, int32_t slot, int64_t *position, int32_t *log_len,
                             uint32_t *flags, ssm_stream_t stream) {
    if (!pool || slot < 0 || slot >= pool->n_slots) return SSM_ERR_INVALID_ARG;
    ssm::GdnDevice dg(pool->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int64_t pos = 0;
    int32_t ll = 0;
    uint32_t fl = 0;
    cudaError_t e = cudaMemcpyAsync(&pos, pool->position + slot, sizeof(pos), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&ll, pool->log_len + slot, sizeof(ll), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&fl, pool->slot_flags + slot, sizeof(fl), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return SSM_ERR_CUDA;
    if (position) *position = pos;
    if (log_len) *log_len = ll;
    if (flags) *flags = fl;
    return SSM_OK;
}

const char *ssm_gdn_last_commit_path(ssm_gdn_pool pool) { return pool ? pool->commit_path : "none"; }

const char *ssm_gdn_last_path(ssm_gdn_pool pool) { return pool ? pool->last_path : "none"; }

ssm_status ssm_gdn_status(ssm_gdn_pool pool, uint32_t *flags_out, int32_t clear, ssm_stream_t stream) {
    if (!pool || !flags_out) return SSM_ERR_INVALID_ARG;
    ssm::GdnDevice dg(pool->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t f = 0;
    cudaError_t e = cudaMemcpyAsync(&f, pool->flags, sizeof(f), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(pool->flags, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return SSM_ERR_CUDA;
    *flags_out = f;
    return SSM_OK;
}

}  // extern "C"
