// ReplaySSM verify with the checkpoint streamed by tensor-map (TMA) copies
// (Why Speculative Decoding Slows Hybrid Mamba Models, The Fix):
//
//   y_j[p] = decay_j (C_j . h_c[p,:]) + sum_{s <= k+j} W[j][s] x_s[p]
//   W[j][s] = exp(A a_{j,s}) dt_s (C_j . B_s)  (+ D for s = k + j)
//   decay_j = exp(A * all dt applied through step token j)
//
// Two kernels per verify call:
//
// replay_group_coef_kernel  one CTA per (request, group): C_j . B_s once
//     for the group's heads, the step's B, x and dt staged after the log (the
//     commit folds them from there), the non-finite check of the step inputs,
//     then per head (one warp) fp64 prefix sums of dt, W and decay_j into pool
//     scratch, and C in fp32.  No state traffic.
//
// verify_replay_tma_kernel  persistent, one CTA per SM.  A producer warp
//     loads each (request, head) item into a shared-memory ring (as many
//     stages as fit, at most eight): the checkpoint as N / 32 tensor-map boxes
//     of 32 columns x P rows in the 128-byte swizzled layout, the head's whole
//     log of x rows as one 3-D box, and C, W, decay_j with bulk copies.  Two
//     groups of four consumer warps take alternate items.  Warp w holds
//     checkpoint columns 32w .. 32w + 31 of its lane's rows (p = lane,
//     lane + 32) in registers, and log tokens 8w .. 8w + 7 of the same rows,
//     then runs the step tokens j: C_j . h_c as packed FMAs with C_j read as a
//     shared-memory broadcast (no cross-lane reduction), plus its share of
//     sum_s W[j][s] x_s.  The four warps' partial outputs meet in shared
//     memory and are summed once per output.
//
// The swizzle: in a box of 128-byte rows starting on a 1024-byte boundary,
// the 16-byte chunk c of row r sits at chunk c ^ (r % 8).  Lanes reading the
// same logical chunk of eight consecutive rows therefore hit eight different
// bank groups.
#include <cuda.h>

#include <algorithm>

#include "ssm_internal.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kGroupWarps = 4;
constexpr int kGroups = 2;
constexpr int kConsumerWarps = kGroups * kGroupWarps;
constexpr int kTmaThreads = (kConsumerWarps + 1) * 32;
constexpr int kCoefThreads = 256;

__host__ __device__ inline uint32_t up16(uint32_t v) { return (v + 15u) & ~15u; }
__host__ __device__ inline int up4(int v) { return (v + 3) & ~3; }

__device__ __forceinline__ void raise_flag(uint32_t *flags, uint32_t *slot_flags, int slot, uint32_t bit) {
    atomicOr(flags, bit);
    if (bit != SSM_FLAG_POISONED_SLOT) atomicOr(slot_flags + slot, kSlotPoisoned);
}

// ------------------------------------------------------------------ coefficients

// 16 bytes of inputs: non-finite test and widening to fp32.
template <typename TI> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static bool nonfinite(uint4 v) {
        return (__vcmpeq2(v.x & 0x7F807F80u, 0x7F807F80u) | __vcmpeq2(v.y & 0x7F807F80u, 0x7F807F80u) |
                __vcmpeq2(v.z & 0x7F807F80u, 0x7F807F80u) | __vcmpeq2(v.w & 0x7F807F80u, 0x7F807F80u)) != 0u;
    }
    __device__ static void widen(uint4 v, float *o) {  // o 16-byte aligned
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            o[2 * q] = __uint_as_float(w[q] << 16);
            o[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
        }
    }
};
template <> struct Vec16<float> {
    static constexpr int n = 4;
    __device__ static bool nonfinite(uint4 v) {
        return ((v.x & 0x7F800000u) == 0x7F800000u) | ((v.y & 0x7F800000u) == 0x7F800000u) |
               ((v.z & 0x7F800000u) == 0x7F800000u) | ((v.w & 0x7F800000u) == 0x7F800000u);
    }
    __device__ static void widen(uint4 v, float *o) {
        *reinterpret_cast<float4 *>(o) = make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                                                     __uint_as_float(v.w));
    }
};

// smem: C [T1][N] | B [mmax][N] | C.B [T1][mmax] | dt per warp [nw][mmax] | prefix sums per warp [nw][mmax] f64
__host__ __device__ inline size_t gcoef_smem_bytes(int T1, int mmax, int N, int nwarps) {
    size_t f = (size_t)T1 * N + (size_t)mmax * N + (size_t)T1 * mmax + (size_t)nwarps * mmax;
    f = (f + 1) & ~(size_t)1;
    return f * 4 + (size_t)nwarps * mmax * 8;
}

// Rows of x, B, C are moved 16 bytes at a time: the launcher checks that
// P and N rows are multiples of 16 bytes and the pointers 16-byte aligned.
template <int N, typename TI>
__global__ void __launch_bounds__(kCoefThreads) replay_group_coef_kernel(const __grid_constant__ StepArgs a) {
    using V = Vec16<TI>;
    constexpr int EV = V::n;          // elements per 16 bytes
    constexpr int NV = N / EV;        // 16-byte vectors per B or C row
    extern __shared__ float4 smem4[];
    const int g = blockIdx.x, i = blockIdx.y;
    const int slot = a.slots[i];
    const int T1 = a.n_tok, H = a.H, P = a.P, hpg = a.hpg;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int wmax = a.wcap - a.t1max, mmax = wmax + T1;
    const int k = a.log_len[slot];
    if ((a.slot_flags[slot] & kSlotPoisoned) || k < 0 || k > wmax) return;  // the streaming kernel reports it
    const int m = k + T1;
    float *sC = reinterpret_cast<float *>(smem4);
    float *sB = sC + (size_t)T1 * N;
    float *sCB = sB + (size_t)mmax * N;
    float *sDt = sCB + (size_t)T1 * mmax;
    size_t off = (size_t)T1 * N + (size_t)mmax * N + (size_t)T1 * mmax + (size_t)nwarps * mmax;
    off = (off + 1) & ~(size_t)1;
    double *sCum = reinterpret_cast<double *>(reinterpret_cast<float *>(smem4) + off);

    const TI *stepC = reinterpret_cast<const TI *>(a.C);
    const TI *stepB = reinterpret_cast<const TI *>(a.B);
    const TI *lB = reinterpret_cast<const TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    TI *wB = reinterpret_cast<TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    bool bad = false;
    float *cf = a.cf + ((size_t)i * a.G + g) * a.t1max * N;
    for (int e = threadIdx.x; e < T1 * NV; e += blockDim.x) {  // C rows, also kept in fp32
        const int j = e / NV, q = e - j * NV;
        const uint4 v = *reinterpret_cast<const uint4 *>(stepC + (((size_t)i * T1 + j) * a.G + g) * N + q * EV);
        bad |= V::nonfinite(v);
        float *o = sC + (size_t)j * N + q * EV;
        V::widen(v, o);
#pragma unroll
        for (int u = 0; u < EV; u += 4)
            *reinterpret_cast<float4 *>(cf + (size_t)j * N + q * EV + u) = *reinterpret_cast<const float4 *>(o + u);
    }
    for (int e = threadIdx.x; e < m * NV; e += blockDim.x) {  // B rows: the log, then the step
        const int s = e / NV, q = e - s * NV;
        uint4 v;
        if (s < k) {
            v = *reinterpret_cast<const uint4 *>(lB + ((size_t)s * a.G + g) * N + q * EV);
        } else {
            v = *reinterpret_cast<const uint4 *>(stepB + (((size_t)i * T1 + (s - k)) * a.G + g) * N + q * EV);
            bad |= V::nonfinite(v);
            *reinterpret_cast<uint4 *>(wB + ((size_t)s * a.G + g) * N + q * EV) = v;  // staged after the log
        }
        V::widen(v, sB + (size_t)s * N + q * EV);
    }
    {  // the step's x of the group's heads (contiguous per token), staged after the log
        const int rv = hpg * P / EV;  // vectors per token
        const TI *sx = reinterpret_cast<const TI *>(a.x);
        TI *wx = reinterpret_cast<TI *>(a.log_x);
        for (int e = threadIdx.x; e < T1 * rv; e += blockDim.x) {
            const int t = e / rv, q = e - t * rv;
            const uint4 v = *reinterpret_cast<const uint4 *>(sx + (((size_t)i * T1 + t) * H + (size_t)g * hpg) * P + q * EV);
            bad |= V::nonfinite(v);
            *reinterpret_cast<uint4 *>(wx + (((size_t)slot * a.wcap + k + t) * H + (size_t)g * hpg) * P + q * EV) = v;
        }
        for (int e = threadIdx.x; e < T1 * hpg; e += blockDim.x) {
            const int t = e / hpg, h = g * hpg + (e - t * hpg);
            const float d = load_dt(a.dt, ((size_t)i * T1 + t) * H + h, a.dt_bf16);
            bad |= !isfinite(d);
            a.log_dt[((size_t)slot * a.wcap + k + t) * H + h] = d;
        }
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }
    for (int pr = threadIdx.x; pr < T1 * m; pr += blockDim.x) {  // C_j . B_s, one thread per pair
        const int j = pr / m, s = pr - j * m;
        float v = 0.f;
        if (s <= k + j) {
            const float4 *c4 = reinterpret_cast<const float4 *>(sC + (size_t)j * N);
            const float4 *b4 = reinterpret_cast<const float4 *>(sB + (size_t)s * N);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll 8
            for (int q = 0; q < N / 4; ++q) {
                const int qq = (q + lane) & (N / 4 - 1);  // lanes start on different banks
                const float4 c = c4[qq], b = b4[qq];
                acc = ffma2(make_float2(c.x, c.y), make_float2(b.x, b.y), acc);
                acc = ffma2(make_float2(c.z, c.w), make_float2(b.z, b.w), acc);
            }
            v = acc.x + acc.y;
        }
        sCB[(size_t)j * mmax + s] = v;
    }
    __syncthreads();
    float *dts = sDt + (size_t)warp * mmax;
    double *cum = sCum + (size_t)warp * mmax;
    for (int hh = warp; hh < hpg; hh += nwarps) {
        const int h = g * hpg + hh;
        const float A = a.A[h], D = a.D[h];
        double carry = 0.0;  // inclusive prefix sums of dt in fp64: their differences lose nothing
        for (int base = 0; base < m; base += 32) {
            const int s = base + lane;
            const float d = s < m ? a.log_dt[((size_t)slot * a.wcap + s) * H + h] : 0.f;
            double v = (double)d;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (s < m) {
                dts[s] = d;
                cum[s] = carry + v;
            }
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        __syncwarp();
        // W rows over the whole stride: zero past k + j, so readers need no bound
        float *wrow = a.wsc + ((size_t)i * H + h) * a.t1max * a.cb_w;
        for (int s = lane; s < a.cb_w; s += 32) {
            const double cs = s < m ? cum[s] : 0.0;
            const float ds = s < m ? dts[s] : 0.f;
            for (int j = 0; j < T1; ++j) {
                float w = 0.f;
                if (s <= k + j) {
                    w = expf(A * (float)(cum[k + j] - cs)) * ds * sCB[(size_t)j * mmax + s];
                    if (s == k + j) w += D;  // skip connection D x_j
                }
                wrow[(size_t)j * a.cb_w + s] = w;
            }
        }
        for (int j = lane; j < T1; j += 32) a.dec[((size_t)i * H + h) * a.t1pad + j] = expf(A * (float)cum[k + j]);
        __syncwarp();
    }
}

// ------------------------------------------------------------------ streaming kernel

constexpr int kMaxStages = 8;
constexpr int kLogPairs = 4;  // log tokens per warp = 2 * kLogPairs, so the log capacity is at most 32

// Byte offsets inside one ring stage, and of the areas after the ring.
struct TmaLayout {
    uint32_t st, xs, cf, w, dec, hdr, stage, red, bars, fixed;
};

__host__ __device__ inline TmaLayout tma_layout(int P, int N, int in_b, int T1, int wcap, int cb_w) {
    TmaLayout L;
    uint32_t o = 0;
    L.st = 0;  o = (uint32_t)P * N * 4;
    L.xs = o;  o = up16(o + (uint32_t)wcap * P * in_b);
    L.cf = o;  o = up16(o + (uint32_t)T1 * N * 4);
    L.w = o;   o = up16(o + (uint32_t)T1 * cb_w * 4);
    L.dec = o; o = up16(o + (uint32_t)up4(T1) * 4);
    L.hdr = o; o += 16;
    L.stage = (o + 1023u) & ~1023u;
    // after the ring (offsets relative to its end): partial sums, barriers
    L.red = 0;
    L.bars = up16((uint32_t)kConsumerWarps * T1 * P * 4);
    L.fixed = L.bars + 2 * kMaxStages * 8 + 1024;  // + slack to align the ring to 1024 bytes
    return L;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                              uint32_t *flags) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && *abort) return false;
    }
    *abort = 1u;
    atomicOr(flags, SSM_FLAG_TIMEOUT);
    return false;
}

// Barrier over one consumer group (named barrier 1 + grp) that ORs a predicate.
__device__ __forceinline__ bool group_or(int grp, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(1 + grp), "r"(kGroupWarps * 32)
        : "memory");
    return r != 0;
}

// RP rows per lane (p = lane, lane + 32); N <= 128, so a warp holds at most
// one 32-column block of the checkpoint in registers.
template <typename TI, int RP>
__global__ void __launch_bounds__(kTmaThreads, 1)
    verify_replay_tma_kernel(const __grid_constant__ StepArgs a, const __grid_constant__ CUtensorMap tm_state,
                             const __grid_constant__ CUtensorMap tm_x, int nstage) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t s_abort;
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int P = a.P, N = a.N, T1 = a.n_tok, H = a.H;
    const int wmax = a.wcap - a.t1max;
    const int nkb = N / 32;
    const TmaLayout L = tma_layout(P, N, (int)sizeof(TI), T1, a.wcap, a.cb_w);
    unsigned char *after = smem + (size_t)nstage * L.stage;
    uint64_t *full = reinterpret_cast<uint64_t *>(after + L.bars);
    uint64_t *empty = full + kMaxStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = a.batch * H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstage; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kGroupWarps);
        }
        mbar_fence_init();
        s_abort = 0u;
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)P * N * 4 + (uint32_t)a.wcap * P * sizeof(TI) + (uint32_t)T1 * N * 4 +
                                   (uint32_t)T1 * a.cb_w * 4 + (uint32_t)up4(T1) * 4;
            int last[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) last[s] = -1;
            for (int u = 0;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int st = u % nstage;
                if (u >= nstage && !wait_or_abort(&empty[st], (uint32_t)((u / nstage) - 1) & 1u, &s_abort, a.flags))
                    break;
                const int i = item / H, h = item - i * H;
                const int slot = a.slots[i];
                const int g = h / a.hpg;
                const int k = a.log_len[slot];
                uint32_t gate = 0;
                if (a.slot_flags[slot] & kSlotPoisoned) gate = SSM_FLAG_POISONED_SLOT;
                else if (k < 0 || k > wmax) gate = SSM_FLAG_BAD_ACCEPT;
                unsigned char *S = smem + (size_t)st * L.stage;
                int *hdr = reinterpret_cast<int *>(S + L.hdr);
                hdr[0] = (int)gate;
                hdr[1] = k;
                if (gate) {
                    mbar_arrive(&full[st]);
                    continue;
                }
                mbar_arrive_expect_tx(&full[st], bytes);
                const int row0 = (slot * H + h) * P;
                for (int kb = 0; kb < nkb; ++kb) tma_load_2d(S + L.st + (size_t)kb * P * 128, &tm_state, kb * 32, row0, &full[st]);
                tma_load_3d(S + L.xs, &tm_x, 0, h, slot * a.wcap, &full[st]);
                bulk_g2s(S + L.cf, a.cf + ((size_t)i * a.G + g) * a.t1max * N, (uint32_t)T1 * N * 4, &full[st]);
                bulk_g2s(S + L.w, a.wsc + ((size_t)i * H + h) * a.t1max * a.cb_w, (uint32_t)T1 * a.cb_w * 4, &full[st]);
                bulk_g2s(S + L.dec, a.dec + ((size_t)i * H + h) * a.t1pad, (uint32_t)up4(T1) * 4, &full[st]);
                last[st] = u;
            }
            // no copy may still be landing when the CTA exits
            for (int s = 0; s < nstage; ++s)
                if (last[s] >= 0 && !mbar_wait(&full[s], (uint32_t)(last[s] / nstage) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int grp = warp / kGroupWarps, w = warp % kGroupWarps, gt = w * 32 + lane;
        float *red = reinterpret_cast<float *>(after + L.red) + (size_t)grp * kGroupWarps * T1 * P;  // [4][T1][P]
        TI *y = reinterpret_cast<TI *>(a.y);
        const int s0 = w * 2 * kLogPairs;  // this warp's log tokens: s0 .. s0 + 2 kLogPairs - 1
        for (int u = grp;; u += kGroups) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            const int st = u % nstage;
            const bool ok = wait_or_abort(&full[st], (uint32_t)(u / nstage) & 1u, &s_abort, a.flags);
            if (group_or(grp, !ok)) break;
            const unsigned char *S = smem + (size_t)st * L.stage;
            const int gate = reinterpret_cast<const int *>(S + L.hdr)[0];
            const int k = reinterpret_cast<const int *>(S + L.hdr)[1];
            const int i = item / H, h = item - i * H;
            if (gate) {
                if (gt == 0) raise_flag(a.flags, a.slot_flags, a.slots[i], (uint32_t)gate);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
                continue;
            }
            const int m = k + T1;
            // this warp's 32 checkpoint columns of rows p = lane + 32 r, into registers
            const bool has_cols = w < nkb;
            float4 hs[8][RP];
            {
                const unsigned char *box = S + L.st + (size_t)w * P * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
#pragma unroll
                    for (int r = 0; r < RP; ++r) {
                        const int p = lane + 32 * r;
                        hs[c][r] = has_cols && p < P
                                       ? *reinterpret_cast<const float4 *>(box + (size_t)p * 128 + ((c ^ (lane & 7)) << 4))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
            }
            // this warp's log tokens as (x_s, x_{s+1}) pairs; zero past the sequence
            const TI *xs = reinterpret_cast<const TI *>(S + L.xs);
            float2 xr[kLogPairs][RP];
#pragma unroll
            for (int q = 0; q < kLogPairs; ++q)
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    const int p = lane + 32 * r, s = s0 + 2 * q;
                    xr[q][r].x = (p < P && s < m) ? to_f(xs[(size_t)s * P + p]) : 0.f;
                    xr[q][r].y = (p < P && s + 1 < m) ? to_f(xs[(size_t)(s + 1) * P + p]) : 0.f;
                }
            const float *cf = reinterpret_cast<const float *>(S + L.cf) + w * 32;
            const float *Ws = reinterpret_cast<const float *>(S + L.w) + s0;
            const float *dec = reinterpret_cast<const float *>(S + L.dec);
            const int npairs = min(kLogPairs, max(0, (m - s0 + 1) >> 1));
            for (int j = 0; j < T1; ++j) {
                float2 a0[RP], a1[RP], lt[RP];
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    a0[r] = make_float2(0.f, 0.f);
                    a1[r] = make_float2(0.f, 0.f);
                    lt[r] = make_float2(0.f, 0.f);
                }
                if (has_cols) {
                    const float4 *cj = reinterpret_cast<const float4 *>(cf + (size_t)j * N);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 cv = cj[c];
#pragma unroll
                        for (int r = 0; r < RP; ++r) {
                            a0[r] = ffma2(make_float2(cv.x, cv.y), make_float2(hs[c][r].x, hs[c][r].y), a0[r]);
                            a1[r] = ffma2(make_float2(cv.z, cv.w), make_float2(hs[c][r].z, hs[c][r].w), a1[r]);
                        }
                    }
                }
                const float *wj = Ws + (size_t)j * a.cb_w;
#pragma unroll
                for (int q = 0; q < kLogPairs; ++q) {
                    if (q < npairs) {
                        const float2 wv = *reinterpret_cast<const float2 *>(wj + 2 * q);
#pragma unroll
                        for (int r = 0; r < RP; ++r) lt[r] = ffma2(wv, xr[q][r], lt[r]);
                    }
                }
                const float dj = dec[j];
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    const int p = lane + 32 * r;
                    if (p < P)
                        red[((size_t)w * T1 + j) * P + p] =
                            fmaf(dj, (a0[r].x + a0[r].y) + (a1[r].x + a1[r].y), lt[r].x + lt[r].y);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);  // the stage is no longer read
            bar_sync_named(1 + grp, kGroupWarps * 32);
            for (int e = gt; e < T1 * P; e += kGroupWarps * 32) {
                const int j = e / P, p = e - j * P;
                const float v = (red[(size_t)j * P + p] + red[((size_t)T1 + j) * P + p]) +
                                (red[((size_t)2 * T1 + j) * P + p] + red[((size_t)3 * T1 + j) * P + p]);
                y[(((size_t)i * T1 + j) * H + h) * P + p] = from_f<TI>(v);
            }
        }
    }
    __syncthreads();
}

template <typename Kernel>
cudaError_t set_smem(Kernel k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

bool replay_tma_encode(Pool &p) {
    p.tm_ok = false;
    if (p.cfg.mode != SSM_MODE_REPLAY) return false;
    if (p.N % 32 != 0 || p.N > 128 || p.P % 8 != 0 || p.P > 64 || p.wcap > 8 * kLogPairs ||
        ((size_t)p.P * p.in_bytes) % 16 != 0)
        return false;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return false;
    using Encode = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    const Encode enc = reinterpret_cast<Encode>(fn);
    // checkpoint: rows (slot, head, p) of N fp32 values; box 32 columns x P rows, 128-byte swizzle
    const cuuint64_t sd[2] = {(cuuint64_t)p.N, (cuuint64_t)p.n_slots * p.H * p.P};
    const cuuint64_t ss[1] = {(cuuint64_t)p.N * 4};
    const cuuint32_t sb[2] = {32u, (cuuint32_t)p.P};
    const cuuint32_t se[2] = {1u, 1u};
    if (enc(&p.tm_state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.state, sd, ss, sb, se, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return false;
    // log x: [slot * wcap + s][head][p]; box = one head's whole log (wcap rows of P)
    const cuuint64_t xd[3] = {(cuuint64_t)p.P, (cuuint64_t)p.H, (cuuint64_t)p.n_slots * p.wcap};
    const cuuint64_t xst[2] = {(cuuint64_t)p.P * p.in_bytes, (cuuint64_t)p.H * p.P * p.in_bytes};
    const cuuint32_t xb[3] = {(cuuint32_t)p.P, 1u, (cuuint32_t)p.wcap};
    const cuuint32_t xe[3] = {1u, 1u, 1u};
    const CUtensorMapDataType xt =
        p.cfg.input_dtype == SSM_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (enc(&p.tm_logx, xt, 3, p.log_x, xd, xst, xb, xe, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    p.tm_ok = true;
    return true;
}

size_t replay_coef_smem_bytes(const Pool &pool, int n_tok) {
    return gcoef_smem_bytes(n_tok, pool.wcap - pool.t1max + n_tok, pool.N, kCoefThreads / 32);
}

cudaError_t launch_verify_replay_tma(const Pool &pool, const StepArgs &a, cudaStream_t s) {
    if (!pool.tm_ok || !a.wsc || !a.cf || !a.dec) return cudaErrorNotSupported;
    const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
    const int in_b = bf ? 2 : 4;
    if (a.N > 128 || a.wcap > 8 * kLogPairs || (a.hpg * a.P * in_b) % 16 || (a.N * in_b) % 16)
        return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(a.x) % 16 || reinterpret_cast<uintptr_t>(a.B) % 16 ||
        reinterpret_cast<uintptr_t>(a.C) % 16)
        return cudaErrorNotSupported;
    const int T1 = a.n_tok;
    const TmaLayout L = tma_layout(a.P, a.N, in_b, T1, a.wcap, a.cb_w);
    const size_t csmem = replay_coef_smem_bytes(pool, T1);
    int dev = 0, max_smem = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int nstage = std::min(kMaxStages, (int)(((long)max_smem - (long)L.fixed) / (long)L.stage));
    if (nstage < 2 || csmem > (size_t)max_smem) return cudaErrorNotSupported;
    const size_t smem = (size_t)nstage * L.stage + L.fixed;

    cudaError_t e = cudaSuccess;
    SSM_DISPATCH_N(a.N, {
        if (bf) {
            auto k = replay_group_coef_kernel<NN, __nv_bfloat16>;
            e = set_smem(k, csmem);
            if (e != cudaSuccess) return e;
            k<<<dim3(a.G, a.batch), kCoefThreads, csmem, s>>>(a);
        } else {
            auto k = replay_group_coef_kernel<NN, float>;
            e = set_smem(k, csmem);
            if (e != cudaSuccess) return e;
            k<<<dim3(a.G, a.batch), kCoefThreads, csmem, s>>>(a);
        }
    });
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    const int n_items = a.batch * a.H;
    const int grid = std::min(n_items, pool.sm_count);
#define SSM_TMA(TI, RP)                                                                                \
    do {                                                                                               \
        auto k = verify_replay_tma_kernel<TI, RP>;                                                     \
        e = set_smem(k, smem);                                                                         \
        if (e != cudaSuccess) return e;                                                                \
        k<<<grid, kTmaThreads, smem, s>>>(a, pool.tm_state, pool.tm_logx, nstage);                     \
    } while (0)
    if (bf) {
        if (a.P <= 32) SSM_TMA(__nv_bfloat16, 1);
        else SSM_TMA(__nv_bfloat16, 2);
    } else {
        if (a.P <= 32) SSM_TMA(float, 1);
        else SSM_TMA(float, 2);
    }
#undef SSM_TMA
    return cudaGetLastError();
}

}  // namespace ssm
