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
//     then per head (one warp) prefix sums of dt as fp32 pairs, W and decay_j into pool
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

#include "pdl.cuh"
#include "ssm_internal.cuh"
#include "tc.cuh"
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

// smem: C [T1][N] | B [mmax][N] | C.B [T1][mmax] | dt per warp [nw][mmax] | prefix sums per warp [nw][mmax] (pairs)
// fp32 C, B, C.B and dt rows, the fp32-pair prefix sums, then (16-byte aligned) the step's x
// of the group's heads as given (xbytes).
__host__ __device__ inline size_t gcoef_x_offset(int T1, int mmax, int N, int nwarps) {
    size_t f = (size_t)T1 * N + (size_t)mmax * N + (size_t)T1 * mmax + (size_t)nwarps * mmax;
    f = (f + 1) & ~(size_t)1;
    return (f * 4 + (size_t)nwarps * mmax * 8 + 15) & ~(size_t)15;
}
// After the step's x: for bf16 inputs C [T1][N] and B [mmax][N] as given (fp32 inputs land in place), then
// the dt of the window's positions for the group's heads [hpg][mmax].
struct GcoefLayout {
    size_t craw, braw, dta, total;
};
__host__ __device__ inline GcoefLayout gcoef_layout(int T1, int mmax, int N, int nwarps, size_t xbytes, int in_b,
                                                    int hpg) {
    GcoefLayout L;
    size_t o = (gcoef_x_offset(T1, mmax, N, nwarps) + xbytes + 15) & ~(size_t)15;
    L.craw = o;
    if (in_b == 2) o += (size_t)T1 * N * 2;
    L.braw = o;
    if (in_b == 2) o += (size_t)mmax * N * 2;
    L.dta = o;
    o += (size_t)hpg * mmax * 4;
    L.total = o;
    return L;
}
__host__ __device__ inline size_t gcoef_smem_bytes(int T1, int mmax, int N, int nwarps, size_t xbytes, int in_b,
                                                   int hpg) {
    return gcoef_layout(T1, mmax, N, nwarps, xbytes, in_b, hpg).total;
}

// Rows of x, B, C are moved 16 bytes at a time: the launcher checks that
// P and N rows are multiples of 16 bytes and the pointers 16-byte aligned.
template <int N, typename TI, bool kFiv>
__global__ void __launch_bounds__(kCoefThreads, 5) replay_group_coef_kernel(const __grid_constant__ StepArgs a) {
    using V = Vec16<TI>;
    constexpr int EV = V::n;          // elements per 16 bytes
    constexpr int NV = N / EV;        // 16-byte vectors per B or C row
    extern __shared__ float4 smem4[];
    // the streaming kernel may be scheduled as CTAs of this one drain; it waits for this grid's
    // completion before it reads anything this kernel writes.  This grid may itself start as the
    // previous commit's last kernel drains: nothing is read before that grid has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int g = blockIdx.x, i = blockIdx.y;
    const int slot = a.slots[i];
    const int T1 = a.n_tok, H = a.H, P = a.P, hpg = a.hpg;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int wmax = a.wcap - a.t1max, mmax = wmax + T1;
    const int kl = a.log_len[slot];
    // fold in verify (kFiv): a log of W or more tokens is folded by this verify (fold_verify_tc_kernel),
    // whose outputs then come from the new checkpoint over the step alone; the step is staged after the
    // log either way, and the commit moves the kept tokens to the end of the (then empty) log
    bool fold_now = false;
    if constexpr (kFiv) {
        fold_now = kl >= a.fold_w && kl <= wmax;
        if (g == 0 && threadIdx.x == 0) {
            a.stage_pos[slot] = kl;
            if (fold_now) a.fv_items[atomicAdd(&a.counts[1], 1)] = make_int2(i, kl);
            else a.plain[atomicAdd(&a.counts[0], 1)] = i;
        }
    }
    if ((a.slot_flags[slot] & kSlotPoisoned) || kl < 0 || kl > wmax) return;  // the streaming kernel reports it
    const int k = fold_now ? 0 : kl;  // logged tokens in the window of the outputs
    const int m = k + T1;
    // log row of window position s (s < k: the log; then the step, staged from row kl)
    auto lrow = [&](int s) { return s < k ? s : kl + (s - k); };
    float *sC = reinterpret_cast<float *>(smem4);
    float *sB = sC + (size_t)T1 * N;
    float *sCB = sB + (size_t)mmax * N;
    size_t off = (size_t)T1 * N + (size_t)mmax * N + (size_t)T1 * mmax + (size_t)nwarps * mmax;
    off = (off + 1) & ~(size_t)1;
    Sum2 *sCum = reinterpret_cast<Sum2 *>(reinterpret_cast<float *>(smem4) + off);
    // the step's x of the group's heads, one contiguous row of hpg P values per token, comes in by
    // bulk copies, is checked here and goes to the log by bulk copies
    __shared__ uint64_t s_xbar;
    TI *sX = reinterpret_cast<TI *>(reinterpret_cast<unsigned char *>(smem4) + gcoef_x_offset(T1, mmax, N, nwarps));
    const uint32_t xrow = (uint32_t)(hpg * P * (int)sizeof(TI));
    const TI *sx = reinterpret_cast<const TI *>(a.x);
    TI *wx = reinterpret_cast<TI *>(a.log_x);
    if (threadIdx.x == 0) {
        mbar_init(&s_xbar, 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(&s_xbar, (uint32_t)T1 * xrow);
        for (int t = 0; t < T1; ++t)
            bulk_g2s(sX + (size_t)t * hpg * P, sx + (((size_t)i * T1 + t) * H + (size_t)g * hpg) * P, xrow, &s_xbar);
    }

    const TI *stepC = reinterpret_cast<const TI *>(a.C);
    const TI *stepB = reinterpret_cast<const TI *>(a.B);
    const TI *lB = reinterpret_cast<const TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    TI *wB = reinterpret_cast<TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    bool bad = false;
    float *cf = a.cf + ((size_t)i * a.G + g) * a.cf_rows * N;
    const int nm = a.cf_nm;
    // bf16 inputs and the tensor-core kernel: C stays bf16, 64 columns per 128-byte row
    const bool bf_op = sizeof(TI) == 2 && nm != 0;
    TI *cfb = reinterpret_cast<TI *>(cf);
    auto cfb_chunk = [&](int j, int n) -> TI * {  // 8 values (a 16-byte chunk) of row j, columns n .. n + 7
        const int kb = n >> 6, c = (n & 63) >> 3;
        return cfb + ((size_t)kb * nm + j) * 64 + ((c ^ (j & 7)) << 3);
    };
    // fp32 C for the streaming kernels: 4 values (a 16-byte chunk) of row j, columns n .. n + 3
    auto cf_chunk = [&](int j, int n) -> float * {
        if (!nm) return cf + (size_t)j * N + n;
        const int kb = n >> 5, c = (n & 31) >> 2;
        return cf + ((size_t)kb * nm + j) * 32 + ((c ^ (j & 7)) << 2);
    };
    // every load of the CTA in flight at once: C and B rows (the log's, then the step's) as 16-byte async
    // copies into shared memory (fp32 inputs straight into place, bf16 beside and widened below), and the
    // dt of the window's positions for the group's heads, the step's checked and staged after the log
    const GcoefLayout GL = gcoef_layout(T1, mmax, N, nwarps, (size_t)T1 * xrow, (int)sizeof(TI), hpg);
    unsigned char *sbytes = reinterpret_cast<unsigned char *>(smem4);
    TI *rC = sizeof(TI) == 2 ? reinterpret_cast<TI *>(sbytes + GL.craw) : reinterpret_cast<TI *>(sC);
    TI *rB = sizeof(TI) == 2 ? reinterpret_cast<TI *>(sbytes + GL.braw) : reinterpret_cast<TI *>(sB);
    float *sDa = reinterpret_cast<float *>(sbytes + GL.dta);  // [hpg][mmax]
    for (int e = threadIdx.x; e < T1 * NV; e += blockDim.x) {
        const int j = e / NV, q = e - j * NV;
        cp_async16(rC + (size_t)j * N + q * EV, stepC + (((size_t)i * T1 + j) * a.G + g) * N + q * EV);
    }
    for (int e = threadIdx.x; e < m * NV; e += blockDim.x) {
        const int s = e / NV, q = e - s * NV;
        cp_async16(rB + (size_t)s * N + q * EV, s < k ? lB + ((size_t)s * a.G + g) * N + q * EV
                                                      : stepB + (((size_t)i * T1 + (s - k)) * a.G + g) * N + q * EV);
    }
    cp_async_commit();
    for (int e = threadIdx.x; e < hpg * m; e += blockDim.x) {
        const int hh = e / m, s = e - hh * m, h = g * hpg + hh;
        float d;
        if (s < k) {
            d = a.log_dt[((size_t)slot * a.wcap + s) * H + h];
        } else {
            d = load_dt(a.dt, ((size_t)i * T1 + (s - k)) * H + h, a.dt_bf16);
            bad |= !isfinite(d);
            a.log_dt[((size_t)slot * a.wcap + kl + (s - k)) * H + h] = d;
        }
        sDa[(size_t)hh * mmax + s] = d;
    }
    cp_async_wait<0>();
    __syncthreads();
    for (int e = threadIdx.x; e < T1 * NV; e += blockDim.x) {  // C rows, also kept in fp32
        const int j = e / NV, q = e - j * NV;
        const uint4 v = *reinterpret_cast<const uint4 *>(rC + (size_t)j * N + q * EV);
        bad |= V::nonfinite(v);
        float *o = sC + (size_t)j * N + q * EV;
        if (sizeof(TI) == 2) V::widen(v, o);
        if (bf_op) {
            *reinterpret_cast<uint4 *>(cfb_chunk(j, q * EV)) = v;
        } else {
#pragma unroll
            for (int u = 0; u < EV; u += 4)
                *reinterpret_cast<float4 *>(cf_chunk(j, q * EV + u)) = *reinterpret_cast<const float4 *>(o + u);
        }
    }
    if (bf_op) {
        for (int e = threadIdx.x; e < (nm - T1) * (N / 8); e += blockDim.x) {  // padding rows of the MMA operand
            const int j = T1 + e / (N / 8), n = (e % (N / 8)) * 8;
            *reinterpret_cast<uint4 *>(cfb_chunk(j, n)) = make_uint4(0u, 0u, 0u, 0u);
        }
    } else {
        for (int e = threadIdx.x; e < (nm - T1) * (N / 4); e += blockDim.x) {
            const int j = T1 + e / (N / 4), n = (e % (N / 4)) * 4;
            *reinterpret_cast<float4 *>(cf_chunk(j, n)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    for (int e = threadIdx.x; e < m * NV; e += blockDim.x) {  // B rows: the log, then the step
        const int s = e / NV, q = e - s * NV;
        const uint4 v = *reinterpret_cast<const uint4 *>(rB + (size_t)s * N + q * EV);
        if (s >= k) {
            bad |= V::nonfinite(v);
            *reinterpret_cast<uint4 *>(wB + ((size_t)lrow(s) * a.G + g) * N + q * EV) = v;  // staged after the log
        }
        if (sizeof(TI) == 2) V::widen(v, sB + (size_t)s * N + q * EV);
    }
    {  // the step's x, once landed: the non-finite check
        __syncthreads();  // the barrier's initialisation is visible to every thread
        if (!mbar_wait(&s_xbar, 0u)) {
            bad = true;
            if (threadIdx.x == 0) atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
        const uint4 *x4 = reinterpret_cast<const uint4 *>(sX);
        for (int e = threadIdx.x; e < T1 * (int)(xrow / 16); e += blockDim.x) bad |= V::nonfinite(x4[e]);
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }
    if (threadIdx.x == 0) {  // x to the log, after the log's k rows; waited for at the end
        for (int t = 0; t < T1; ++t)
            bulk_s2g(wx + (((size_t)slot * a.wcap + kl + t) * H + (size_t)g * hpg) * P, sX + (size_t)t * hpg * P, xrow);
        bulk_commit();
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
    Sum2 *cum = sCum + (size_t)warp * mmax;
    for (int hh = warp; hh < hpg; hh += nwarps) {
        const int h = g * hpg + hh;
        const float A = a.A[h], D = a.D[h];
        const float *dts = sDa + (size_t)hh * mmax;
        warp_prefix_sum2(dts, cum, m, lane);  // differences of these are exact to fp32
        __syncwarp();
        // W rows over the whole stride: zero past k + j, so readers need no bound
        float *wrow = a.wsc + ((size_t)i * H + h) * a.t1max * a.cb_w;
        for (int s = lane; s < a.cb_w; s += 32) {
            const Sum2 cs = s < m ? cum[s] : Sum2{0.f, 0.f};
            const float ds = s < m ? dts[s] : 0.f;
            for (int j = 0; j < T1; ++j) {
                float w = 0.f;
                if (s <= k + j) {
                    w = expf(A * sum2_diff(cum[k + j], cs)) * ds * sCB[(size_t)j * mmax + s];
                    if (s == k + j) w += D;  // skip connection D x_j
                }
                wrow[(size_t)j * a.cb_w + s] = w;
            }
        }
        for (int j = lane; j < T1; j += 32) a.dec[((size_t)i * H + h) * a.t1pad + j] = expf(A * (cum[k + j].hi + cum[k + j].lo));
        __syncwarp();
    }
    if (threadIdx.x == 0) bulk_wait0();  // the log's x rows are written before the CTA ends
}

// ------------------------------------------------------------------ streaming kernel

constexpr int kMaxStages = 8;
constexpr int kLogPairs = 4;  // log tokens per warp = 2 * kLogPairs, so the log capacity is at most 32
constexpr int kMaxTmaLog = 64;  // log capacity the tensor-core kernel and the fold take (a box is <= 256 rows)

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
        // The whole warp walks the items; lanes prefetch the gate inputs (log
        // length, slot flags) of the next 32 items, lane 0 issues the copies.
        const uint32_t bytes = (uint32_t)P * N * 4 + (uint32_t)a.wcap * P * sizeof(TI) + (uint32_t)T1 * N * 4 +
                               (uint32_t)T1 * a.cb_w * 4 + (uint32_t)up4(T1) * 4;
        int last[kMaxStages];
        for (int s = 0; s < kMaxStages; ++s) last[s] = -1;
        int my_k = 0;
        uint32_t my_gate = 0;
        for (int u = 0;; ++u) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            if ((u & 31) == 0) {
                const int it2 = item + lane * gridDim.x;
                my_k = 0;
                my_gate = 0;
                if (it2 < n_items) {
                    const int sl = a.slots[it2 / H];
                    my_k = a.log_len[sl];
                    if (a.slot_flags[sl] & kSlotPoisoned) my_gate = SSM_FLAG_POISONED_SLOT;
                    else if (my_k < 0 || my_k > wmax) my_gate = SSM_FLAG_BAD_ACCEPT;
                }
            }
            const int k = __shfl_sync(0xffffffffu, my_k, u & 31);
            const uint32_t gate = __shfl_sync(0xffffffffu, my_gate, u & 31);
            const int st = u % nstage;
            int ok = 1;
            if (u >= nstage && lane == 0)
                ok = wait_or_abort(&empty[st], (uint32_t)((u / nstage) - 1) & 1u, &s_abort, a.flags);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (lane == 0) {
                const int i = item / H, h = item - i * H;
                const int slot = a.slots[i];
                const int g = h / a.hpg;
                unsigned char *S = smem + (size_t)st * L.stage;
                int *hdr = reinterpret_cast<int *>(S + L.hdr);
                hdr[0] = (int)gate;
                hdr[1] = k;
                if (gate) {
                    mbar_arrive(&full[st]);
                } else {
                    mbar_arrive_expect_tx(&full[st], bytes);
                    const int row0 = (slot * H + h) * P;
                    for (int kb = 0; kb < nkb; ++kb)
                        tma_load_2d(S + L.st + (size_t)kb * P * 128, &tm_state, kb * 32, row0, &full[st]);
                    tma_load_3d(S + L.xs, &tm_x, 0, h, slot * a.wcap, &full[st]);
                    bulk_g2s(S + L.cf, a.cf + ((size_t)i * a.G + g) * a.cf_rows * N, (uint32_t)T1 * N * 4, &full[st]);
                    bulk_g2s(S + L.w, a.wsc + ((size_t)i * H + h) * a.t1max * a.cb_w, (uint32_t)T1 * a.cb_w * 4,
                             &full[st]);
                    bulk_g2s(S + L.dec, a.dec + ((size_t)i * H + h) * a.t1pad, (uint32_t)up4(T1) * 4, &full[st]);
                    last[st] = u;
                }
            }
            __syncwarp();
        }
        // no copy may still be landing when the CTA exits
        if (lane == 0)
            for (int s = 0; s < nstage; ++s)
                if (last[s] >= 0 && !mbar_wait(&full[s], (uint32_t)(last[s] / nstage) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
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

// ------------------------------------------------------------------ tensor-core streaming kernel
//
// verify_replay_tc_kernel: the same outputs with C_j . h_c on the 5th-generation
// tensor cores.  An item is the pair of heads (h, h + 1) of one request (same
// group, so the same C): their checkpoints stacked are the M = 128 rows of A
// (P = 64 each), K = N, and the step tokens are the N = NM columns (16 or 32,
// padded).  A kind::tf32 MMA reads an fp32 operand through its tf32 part: the
// sign, the exponent and the top 10 mantissa bits (the 13 low bits are
// dropped).  With hi = v with those 13 bits cleared and lo = v - hi (exact in
// fp32, at most 2^-10 |v|, and itself cut to tf32 with a relative error of
// 2^-11 more), C . h = C . h_hi + C . h_lo, and for fp32 inputs also
// + C_lo . h_hi; bf16 C is a tf32 value already.  The dropped C_lo . h_lo and
// the cut of lo leave about 2^-20 of each product, below the fp32 rounding of
// the sum.
//
// Data flow per item: one producer streams the checkpoint in 32-column blocks
// (16 KiB: 128 rows x 128 bytes, 128-byte swizzle) into a ring of slots, as far
// ahead as the ring allows; another loads C (fp32, K-major swizzled), the x
// rows, W and decay_j of the two heads into a small per-item ring.  Only those
// two rings pace the loads: the checkpoint of an item is in flight while earlier
// items are still in the MMA and the epilogue.  Each split warp reads its 32 rows of a block (thread =
// row, so the swizzle spreads the eight rows of a bank group), writes hi and
// lo into a 64-column TMEM operand slot and frees the ring slot at once; the
// warps work independently (no barrier between them per block).  The MMA
// issuer takes A (hi, then lo) from TMEM and B (C) from shared memory, one
// accumulator per item, and commits once per item (a commit costs about as
// much as four MMAs) to that item's `done` barrier, which frees its operand
// slots and stage and hands D to the epilogue.  Split and MMA treat every item
// alike; an item whose request is gated (poisoned slot, bad accept count) gets
// no per-item loads and the epilogue drops its D.
//
// Warps:  0-3 epilogue (TMEM lane quarters 0-3: row = 32 q + lane, q = w % 4),
//         the log term from the staged x and W rows, y = decay_j D[row][j] +
//         log term; with 16 step columns a second epilogue group (warps 16-19)
//         takes the odd items, since one group's time per item (log term,
//         D read, stores) is longer than the checkpoint stream's;
//         4-7 and 8-11 split, two groups (each over the four lane quarters)
//           taking even and odd blocks: a block takes a group about half a
//           microsecond end to end, so one group alone could not keep up with
//           the stream; group 0 also makes C_lo for fp32 inputs;
//         12 per-item producer (gate inputs prefetched a warp at a time);
//         13 checkpoint producer;
//         14, 15 MMA issuers (lane 0), taking alternate items, since an issuer's
//           waits on its barriers take about as long as its MMAs; 14 owns TMEM.
// TMEM: D buffer b (four) at columns NM b; operand slots of 64 columns (hi at
// +0, lo at +32) from column 4 NM.
constexpr int kTcEpiWarps = 4;
constexpr int kTcSplitGroups = 2;  // split groups take alternate checkpoint blocks
constexpr int kTcProd = 4 + 4 * kTcSplitGroups;
constexpr int kTcRing = kTcProd + 1;
constexpr int kTcMma = kTcRing + 1;  // and kTcMma + 1: two issuers taking alternate items
constexpr int kTcMmaWarps = 2;
constexpr int kTcMaxRing = 12;  // checkpoint blocks in flight
constexpr int kTcMaxAux = 4;    // per-item stages, an even count: stage u % naux then serves items of one
                                // parity, i.e. one MMA issuer and one epilogue group, and each of them
                                // sees every phase of its stages' barriers in order
constexpr int kTcMaxASlots = 12;  // TMEM operand slots, hi + lo of one 32-column block each (see TcOperand)
constexpr int kTcDone = 4;      // per-item MMA completion barriers (waiters lag by < 4 items)
constexpr int kTcDbuf = 4;      // TMEM accumulators: the MMA runs at most 4 items ahead of the epilogue
constexpr uint32_t kTcCols = 512;
constexpr uint32_t kTf32Keep = 0xFFFFE000u;  // sign, exponent and the 10 tf32 mantissa bits

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) { return *reinterpret_cast<const uint32_t *>(&v); }
static_assert(kTcDbuf <= kTcDone, "a done barrier must not complete twice ahead of its waiter");
static_assert(kTcMaxAux % 2 == 0 && kTcDbuf % kTcMmaWarps == 0 && kTcDone % kTcMmaWarps == 0,
              "a barrier indexed by item must serve items of one issuer");

// The product C . h_c per input type.  fp32 inputs: kind::tf32, h_c as tf32 hi
// + lo in 64 TMEM columns per block (32-bit elements), C fp32 (32 per 128-byte
// row) and its remainder C_lo.  bf16 inputs: kind::f16 (K = 16 per MMA, half
// the MMAs), h_c as bf16 hi = rn(v) and lo = rn(v - hi), which carry 16
// significant bits (|v - hi - lo| <= 2^-17 |v|, far below the bf16 rounding of
// y), packed two per column in 32 TMEM columns per block; C bf16 as given (64
// per 128-byte row).
template <typename TI>
struct TcOperand {
    static constexpr bool kF16 = sizeof(TI) == 2;
    static constexpr int kSlotCols = kF16 ? 32 : 64;
    static constexpr int kSlots = 384 / kSlotCols;
    static constexpr int kRowElems = kF16 ? 64 : 32;  // C elements per 128-byte operand row
};
static_assert(TcOperand<float>::kSlots <= kTcMaxASlots && TcOperand<__nv_bfloat16>::kSlots <= kTcMaxASlots, "");

// One epilogue group per item, alternating when there are two (group_or groups 0 and 1).
template <int NM>
struct TcShape {
    static constexpr int kEpiGroups = NM == 16 ? 2 : 1;
    static constexpr int kThreads = (kTcMma + kTcMmaWarps + 4 * (kEpiGroups - 1)) * 32;
};

struct TcLayout {
    uint32_t Bt, Blo, xs, w, dec, hdr, aux;  // inside one per-item stage
    uint32_t ring_bytes, aux_base, bars;     // after alignment of the base to 1024
};

__host__ __device__ inline TcLayout tc_layout(int N, int NM, int P, int in_b, int wcap, int t1max, int cb_w,
                                             int t1pad, bool split_c, int nring, int naux) {
    TcLayout L;
    const uint32_t nkb = (uint32_t)(N * in_b) / 128u;      // 128-byte column blocks of C
    uint32_t o = 0;
    L.Bt = 0;   o = nkb * (uint32_t)NM * 128u;            // NM rows x 128 bytes per column block
    L.Blo = o;  if (split_c) o += nkb * (uint32_t)NM * 128u;
    L.xs = o;   o = up16(o + 2u * wcap * P * in_b);       // [s][2 heads][P]
    L.w = o;    o = up16(o + 2u * t1max * cb_w * 4);      // [2 heads][t1max][cb_w]
    L.dec = o;  o = up16(o + 2u * t1pad * 4);             // [2 heads][t1pad]
    L.hdr = o;  o += 16;
    L.aux = (o + 1023u) & ~1023u;
    L.ring_bytes = (uint32_t)nring * 16384u;
    L.aux_base = L.ring_bytes;
    L.bars = L.aux_base + (uint32_t)naux * L.aux;
    return L;
}

__host__ __device__ inline size_t tc_smem_bytes(const TcLayout &L) {
    return (size_t)L.bars + (2 * kTcMaxRing + 2 * kTcMaxAux + kTcMaxASlots + kTcDone + kTcDbuf) * 8 + 1024;
}

template <typename TI, int NM, bool kList>
__global__ void __launch_bounds__(TcShape<NM>::kThreads, 1)
    verify_replay_tc_kernel(const __grid_constant__ StepArgs a, const __grid_constant__ CUtensorMap tm_state2,
                            const __grid_constant__ CUtensorMap tm_x2, int nring, int naux) {
    constexpr bool kSplitC = sizeof(TI) == 4;
    using Op = TcOperand<TI>;
    constexpr int AS = Op::kSlots, SWC = Op::kSlotCols;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t s_abort, s_tmem;
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int P = a.P, N = a.N, T1 = a.n_tok, H = a.H;
    const int nkb = N / 32, hp = H / 2;
    const int wmax = a.wcap - a.t1max;
    const TcLayout L = tc_layout(N, NM, P, (int)sizeof(TI), a.wwin, a.t1max, a.cb_w, a.t1pad, kSplitC, nring, naux);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *rfull = bars, *rempty = rfull + kTcMaxRing;                // checkpoint ring
    uint64_t *xfull = rempty + kTcMaxRing, *xempty = xfull + kTcMaxAux;  // per-item ring
    uint64_t *afull = xempty + kTcMaxAux;                                // TMEM operand slots
    uint64_t *done = afull + kTcMaxASlots;                               // MMAs of an item finished
    uint64_t *dempty = done + kTcDone;                                   // TMEM D buffers
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nring; ++s) {
            mbar_init(&rfull[s], 1);
            mbar_init(&rempty[s], 4);
        }
        for (int s = 0; s < naux; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], kTcEpiWarps);
        }
        for (int s = 0; s < AS; ++s) mbar_init(&afull[s], 4);
        for (int s = 0; s < kTcDone; ++s) mbar_init(&done[s], 1);
        for (int s = 0; s < kTcDbuf; ++s) mbar_init(&dempty[s], kTcEpiWarps);
        mbar_fence_init();
        s_abort = 0u;
    }
    if (warp == kTcMma) tc::tmem_alloc(&s_tmem, kTcCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    // kList (the verify folds full logs): the coefficient kernel lists the other requests; every role
    // reads the list, so every role waits for that kernel (else only the per-item producer does)
    int n_items = a.batch * hp;
    if constexpr (kList) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        n_items = *(volatile const int32_t *)&a.counts[0] * hp;
    }
    auto request = [&](int item) {
        if constexpr (kList) return a.plain[item / hp];
        else return item / hp;
    };

    if (warp == kTcProd) {
        // ------------------------------------------------------------ producer
        const uint32_t cbytes = (uint32_t)(N / Op::kRowElems) * NM * 128u;  // C, already in the operand layout
        const uint32_t xbytes = cbytes + 2u * a.wwin * P * sizeof(TI) + 2u * a.t1max * a.cb_w * 4u + 2u * a.t1pad * 4u;
        int xlast[kTcMaxAux];
        for (int s = 0; s < kTcMaxAux; ++s) xlast[s] = -1;
        // C in the operand layout, W, decay_j, the staged log rows and the slot flags come from the
        // coefficient kernel, launched just before this one
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int my_k = 0;
        uint32_t my_gate = 0;
        bool alive = true;
        for (int u = 0; alive; ++u) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            if ((u & 31) == 0) {
                const int it2 = item + lane * gridDim.x;
                my_k = 0;
                my_gate = 0;
                if (it2 < n_items) {
                    const int sl = a.slots[request(it2)];
                    my_k = a.log_len[sl];
                    if (a.slot_flags[sl] & kSlotPoisoned) my_gate = SSM_FLAG_POISONED_SLOT;
                    else if (my_k < 0 || my_k > wmax) my_gate = SSM_FLAG_BAD_ACCEPT;
                }
            }
            const int k = __shfl_sync(0xffffffffu, my_k, u & 31);
            const uint32_t gate = __shfl_sync(0xffffffffu, my_gate, u & 31);
            if (lane == 0) {
                const int xs_ = u % naux;
                const int i = request(item), h0 = 2 * (item % hp);
                const int slot = a.slots[i];
                const int g = h0 / a.hpg;
                if (u >= naux && !wait_or_abort(&xempty[xs_], (uint32_t)((u / naux) - 1) & 1u, &s_abort, a.flags)) {
                    alive = false;
                } else {
                    unsigned char *X = smem + L.aux_base + (size_t)xs_ * L.aux;
                    int *hdr = reinterpret_cast<int *>(X + L.hdr);
                    hdr[0] = (int)gate;
                    hdr[1] = k;
                    if (a.test_stall && blockIdx.x == 0 && u == 0) {
                        // tests of the failure path: this item's loads are withheld, so the waits on them
                        // run out and every role of this CTA leaves through its abort path
                    } else if (gate) {
                        mbar_arrive(&xfull[xs_]);
                    } else {
                        mbar_arrive_expect_tx(&xfull[xs_], xbytes);
                        bulk_g2s(X + L.Bt, a.cf + ((size_t)i * a.G + g) * a.cf_rows * N, cbytes, &xfull[xs_]);
                        tma_load_3d(X + L.xs, &tm_x2, 0, h0, slot * a.wcap, &xfull[xs_]);
                        bulk_g2s(X + L.w, a.wsc + ((size_t)i * H + h0) * a.t1max * a.cb_w,
                                 2u * a.t1max * a.cb_w * 4u, &xfull[xs_]);
                        bulk_g2s(X + L.dec, a.dec + ((size_t)i * H + h0) * a.t1pad, 2u * a.t1pad * 4u, &xfull[xs_]);
                        xlast[xs_] = u;
                    }
                }
            }
            alive = __shfl_sync(0xffffffffu, (int)alive, 0) != 0;
        }
        if (lane == 0) {  // no copy may still be landing when the CTA exits
            for (int s = 0; s < naux; ++s)
                if (xlast[s] >= 0 && !mbar_wait(&xfull[s], (uint32_t)(xlast[s] / naux) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp == kTcRing) {
        // ------------------------------------------------------------ checkpoint producer
        if (lane == 0) {
            int rlast[kTcMaxRing];
            for (int s = 0; s < kTcMaxRing; ++s) rlast[s] = -1;
            int nblk = 0;
            bool alive = true;
            for (int u = 0; alive; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int i = request(item), h0 = 2 * (item % hp);
                const int row0 = (a.slots[i] * H + h0) * P;
                for (int kb = 0; kb < nkb; ++kb, ++nblk) {
                    const int rs = nblk % nring;
                    if (nblk >= nring &&
                        !wait_or_abort(&rempty[rs], (uint32_t)((nblk / nring) - 1) & 1u, &s_abort, a.flags)) {
                        alive = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&rfull[rs], 16384u);
                    tma_load_2d(smem + (size_t)rs * 16384, &tm_state2, kb * 32, row0, &rfull[rs]);
                    rlast[rs] = nblk;
                }
            }
            // no copy may still be landing when the CTA exits
            for (int s = 0; s < nring; ++s)
                if (rlast[s] >= 0 && !mbar_wait(&rfull[s], (uint32_t)(rlast[s] / nring) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp >= kTcMma && warp < kTcMma + kTcMmaWarps) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = Op::kF16 ? tc::idesc_bf16_f32(128, NM) : tc::idesc_tf32_f32(128, NM);
            // every item goes through the MMA, so its position u is also its count of items before it
            int last = -1;
            bool alive = true;
            for (int u = warp - kTcMma; alive; u += kTcMmaWarps) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int nproc = u;
                const int xs_ = u % naux;
                if (!wait_or_abort(&xfull[xs_], (uint32_t)(u / naux) & 1u, &s_abort, a.flags)) break;
                const unsigned char *X = smem + L.aux_base + (size_t)xs_ * L.aux;
                const int db = nproc % kTcDbuf;
                if (nproc >= kTcDbuf &&
                    !wait_or_abort(&dempty[db], (uint32_t)((nproc / kTcDbuf) - 1) & 1u, &s_abort, a.flags))
                    break;
                tc::fence_after_sync();
                const uint32_t d_tm = tmem + (uint32_t)db * NM;
                const uint32_t b_hi = smem_addr(X + L.Bt), b_lo = smem_addr(X + L.Blo);
                for (int kb = 0; kb < nkb; ++kb) {
                    const int c = nproc * nkb + kb, as = c % AS;
                    if (!wait_or_abort(&afull[as], (uint32_t)(c / AS) & 1u, &s_abort, a.flags)) {
                        if (kb > 0) {  // MMAs of this item are in flight: let them finish first
                            tc::mma_commit(&done[nproc % kTcDone]);
                            mbar_wait(&done[nproc % kTcDone], (uint32_t)(nproc / kTcDone) & 1u);
                        }
                        alive = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t a_hi = tmem + (uint32_t)kTcDbuf * NM + (uint32_t)as * SWC;
                    if constexpr (Op::kF16) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {  // K = 16 bf16 per MMA: 8 columns of hi (+0) and lo (+16)
                            const uint32_t boff = (uint32_t)(kb >> 1) * NM * 128 + (kb & 1) * 64 + 32 * kk;
                            const uint64_t dbh = tc::smem_desc_sw128(b_hi + boff, 1024);
                            tc::mma_bf16_ta(d_tm, a_hi + 8 * kk, dbh, idesc, (kb | kk) != 0);
                            tc::mma_bf16_ta(d_tm, a_hi + 16 + 8 * kk, dbh, idesc, true);
                        }
                    } else {
                        const uint32_t a_lo = a_hi + 32u;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {  // K = 8 tf32 per MMA
                            const uint32_t boff = (uint32_t)kb * NM * 128 + 32 * kk;
                            const uint64_t dbh = tc::smem_desc_sw128(b_hi + boff, 1024);
                            tc::mma_tf32_ta(d_tm, a_hi + 8 * kk, dbh, idesc, (kb | kk) != 0);
                            tc::mma_tf32_ta(d_tm, a_lo + 8 * kk, dbh, idesc, true);
                            if (kSplitC) tc::mma_tf32_ta(d_tm, a_hi + 8 * kk, tc::smem_desc_sw128(b_lo + boff, 1024), idesc, true);
                        }
                    }
                }
                if (!alive) break;
                tc::mma_commit(&done[nproc % kTcDone]);
                last = u;
            }
            // every MMA this thread issued has completed before TMEM is released (an item cut short
            // above was waited for there; the items before it end with this thread's last commit)
            if (last >= 0 && !mbar_wait(&done[last % kTcDone], (uint32_t)(last / kTcDone) & 1u))
                atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp >= kTcEpiWarps && warp < kTcProd) {
        // ------------------------------------------------------------ split
        const int q = warp & 3;                       // TMEM lane quarter
        const int sg = (warp - kTcEpiWarps) >> 2;     // split group: blocks c with c % 2 == sg
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        int nproc = 0;
        bool alive = true;
        for (int u = 0; alive; ++u) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            if (kSplitC && sg == 0) {  // C_lo = C - C_hi beside C (this warp's share), before block 0 is signalled
                const int xs_ = u % naux;
                if (!wait_or_abort(&xfull[xs_], (uint32_t)(u / naux) & 1u, &s_abort, a.flags)) break;
                unsigned char *X = smem + L.aux_base + (size_t)xs_ * L.aux;
                const uint4 *b4 = reinterpret_cast<const uint4 *>(X + L.Bt);
                uint4 *bl4 = reinterpret_cast<uint4 *>(X + L.Blo);
                for (int e = row; e < nkb * NM * 8; e += 128) {
                    const uint4 v = b4[e];
                    bl4[e] = make_uint4(__float_as_uint(__uint_as_float(v.x) - __uint_as_float(v.x & kTf32Keep)),
                                        __float_as_uint(__uint_as_float(v.y) - __uint_as_float(v.y & kTf32Keep)),
                                        __float_as_uint(__uint_as_float(v.z) - __uint_as_float(v.z & kTf32Keep)),
                                        __float_as_uint(__uint_as_float(v.w) - __uint_as_float(v.w & kTf32Keep)));
                }
                tc::fence_proxy_async_smem();
            }
            for (int kb = 0; kb < nkb; ++kb) {
                const int c = nproc * nkb + kb, rs = c % nring, as = c % AS;
                if ((c & 1) != sg) continue;
                bool ok = wait_or_abort(&rfull[rs], (uint32_t)(c / nring) & 1u, &s_abort, a.flags);
                if (ok && c >= AS) {  // the slot's previous block belongs to item (c - slots) / nkb
                    const int pj = (c - AS) / nkb;
                    ok = wait_or_abort(&done[pj % kTcDone], (uint32_t)(pj / kTcDone) & 1u, &s_abort, a.flags);
                }
                if (!ok) {
                    alive = false;
                    break;
                }
                tc::fence_after_sync();
                // this thread's row of the block: 8 chunks of 16 bytes, chunk c at c ^ (row % 8)
                const unsigned char *blk = smem + (size_t)rs * 16384 + (size_t)row * 128;
                const uint32_t a_hi = tmem + lane_off + (uint32_t)kTcDbuf * NM + (uint32_t)as * SWC;
                if constexpr (Op::kF16) {
                    uint32_t hl[32];  // columns 0-15: hi of elements (2c, 2c + 1); 16-31: lo of the same
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const float4 v = *reinterpret_cast<const float4 *>(blk + ((ch ^ (row & 7)) << 4));
                        const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
                        const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - __low2float(h0), v.y - __high2float(h0));
                        const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - __low2float(h1), v.w - __high2float(h1));
                        hl[2 * ch] = bf2_bits(h0);
                        hl[2 * ch + 1] = bf2_bits(h1);
                        hl[16 + 2 * ch] = bf2_bits(l0);
                        hl[16 + 2 * ch + 1] = bf2_bits(l1);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&rempty[rs]);  // the rows are in registers: free the ring slot
                    tc::tmem_st32(a_hi, hl);
                } else {
                    uint32_t hi[32], lo[32];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(blk + ((ch ^ (row & 7)) << 4));
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            hi[4 * ch + e] = w[e] & kTf32Keep;
                            lo[4 * ch + e] = __float_as_uint(__uint_as_float(w[e]) - __uint_as_float(hi[4 * ch + e]));
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&rempty[rs]);
                    tc::tmem_st32(a_hi, hi);
                    tc::tmem_st32(a_hi + 32u, lo);
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&afull[as]);
            }
            ++nproc;
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 0-3, 16-19)
        constexpr int EG = TcShape<NM>::kEpiGroups;
        const int eg = warp < kTcEpiWarps ? 0 : 1;
        const int q = warp & 3, r = q * 32 + lane, hd = r / 64, p = r - hd * 64;
        TI *y = reinterpret_cast<TI *>(a.y);
        for (int u = eg;; u += EG) {  // every item goes through the MMA, so item u has D buffer u % kTcDbuf
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            const int xs_ = u % naux;
            const bool ok = wait_or_abort(&xfull[xs_], (uint32_t)(u / naux) & 1u, &s_abort, a.flags);
            if (group_or(eg, !ok)) break;
            const unsigned char *X = smem + L.aux_base + (size_t)xs_ * L.aux;
            const int gate = reinterpret_cast<const int *>(X + L.hdr)[0];
            const int k = reinterpret_cast<const int *>(X + L.hdr)[1];
            const int i = request(item), h0 = 2 * (item % hp);
            if (gate && r == 0) raise_flag(a.flags, a.slot_flags, a.slots[i], (uint32_t)gate);
            const int m = gate ? 0 : k + T1;
            // log term sum_s W[j][s] x_s[p], s in quads (the W rows, zero past s = k + j, as float4),
            // every j per quad so that the loads of a quad are independent; cut at the length m
            const int nq = (m + 3) >> 2;
            const TI *xrow = reinterpret_cast<const TI *>(X + L.xs) + (size_t)hd * P + p;  // x_s at s * 2P
            const float *Wh = reinterpret_cast<const float *>(X + L.w) + (size_t)hd * a.t1max * a.cb_w;
            const float *dh = reinterpret_cast<const float *>(X + L.dec) + (size_t)hd * a.t1pad;
            float2 acc[NM];
#pragma unroll
            for (int j = 0; j < NM; ++j) acc[j] = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int qq = 0; qq < nq; ++qq) {
                const int s = 4 * qq;
                const float2 x01 = make_float2(s < m ? to_f(xrow[(size_t)s * 2 * P]) : 0.f,
                                               s + 1 < m ? to_f(xrow[(size_t)(s + 1) * 2 * P]) : 0.f);
                const float2 x23 = make_float2(s + 2 < m ? to_f(xrow[(size_t)(s + 2) * 2 * P]) : 0.f,
                                               s + 3 < m ? to_f(xrow[(size_t)(s + 3) * 2 * P]) : 0.f);
                const float4 *w4 = reinterpret_cast<const float4 *>(Wh) + qq;
#pragma unroll
                for (int j = 0; j < NM; ++j) {
                    if (j < T1) {
                        const float4 wv = w4[(size_t)j * (a.cb_w / 4)];
                        acc[j] = ffma2(make_float2(wv.x, wv.y), x01, acc[j]);
                        acc[j] = ffma2(make_float2(wv.z, wv.w), x23, acc[j]);
                    }
                }
            }
            float lt[NM], dj[NM];
#pragma unroll
            for (int j = 0; j < NM; ++j) {
                lt[j] = acc[j].x + acc[j].y;
                dj[j] = (j < T1 && !gate) ? dh[j] : 0.f;
            }
            const int db = u % kTcDbuf;
            const bool okd = wait_or_abort(&done[u % kTcDone], (uint32_t)(u / kTcDone) & 1u, &s_abort, a.flags);
            if (group_or(eg, !okd)) break;
            __syncwarp();  // the item's MMAs are done with C and the stage is read: hand it back
            if (lane == 0) mbar_arrive(&xempty[xs_]);
            tc::fence_after_sync();
            float d[NM];
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)db * NM;
#pragma unroll
            for (int c = 0; c < NM; c += 16) {
                float part[16];
                tc::tmem_ld16(taddr + c, part);
#pragma unroll
                for (int q = 0; q < 16; ++q) d[c + q] = part[q];
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dempty[db]);
            TI *yrow = y + ((size_t)i * T1 * H + h0 + hd) * P + p;
            if (!gate) {
#pragma unroll
                for (int j = 0; j < NM; ++j)
                    if (j < T1) yrow[(size_t)j * H * P] = from_f<TI>(fmaf(dj[j], d[j], lt[j]));
            }
        }
    }
    __syncwarp();  // warps whose lane 0 ran a role alone arrive at the block barrier converged
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kTcMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTcCols);
    }
}

template <typename Kernel>
cudaError_t set_smem(Kernel k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

TensorMapEncode tensor_map_encoder() {
    static const TensorMapEncode enc = []() -> TensorMapEncode {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<TensorMapEncode>(fn);
    }();
    return enc;
}

bool replay_tma_encode(Pool &p) {
    p.tm_ok = p.tm_tc_ok = p.tm_fold_ok = false;
    p.fold_kp = 0;
    if (p.cfg.mode != SSM_MODE_REPLAY) return false;
    if (p.N % 32 != 0 || p.N > 128 || p.P % 8 != 0 || p.P > 64 || p.wcap > kMaxTmaLog ||
        ((size_t)p.P * p.in_bytes) % 16 != 0)
        return false;
    const TensorMapEncode enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t sd[2] = {(cuuint64_t)p.N, (cuuint64_t)p.n_slots * p.H * p.P};
    const cuuint64_t ss[1] = {(cuuint64_t)p.N * 4};
    const cuuint32_t se[2] = {1u, 1u};
    const cuuint64_t xd[3] = {(cuuint64_t)p.P, (cuuint64_t)p.H, (cuuint64_t)p.n_slots * p.wcap};
    const cuuint64_t xst[2] = {(cuuint64_t)p.P * p.in_bytes, (cuuint64_t)p.H * p.P * p.in_bytes};
    const cuuint32_t xe[3] = {1u, 1u, 1u};
    const CUtensorMapDataType xt =
        p.cfg.input_dtype == SSM_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    // CUDA-core kernel (it holds the log's x rows in registers, so the log capacity is at most 32):
    // checkpoint rows (slot, head, p) of N fp32 values, box 32 columns x P rows, 128-byte swizzle;
    // log x [slot * wcap + s][head][p], box = one head's whole log (wcap rows of P)
    if (p.wcap <= 8 * kLogPairs) {
        const cuuint32_t sb[2] = {32u, (cuuint32_t)p.P};
        const cuuint32_t xb[3] = {(cuuint32_t)p.P, 1u, (cuuint32_t)p.wcap};
        p.tm_ok = enc(&p.tm_state, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.state, sd, ss, sb, se,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
                  enc(&p.tm_logx, xt, 3, p.log_x, xd, xst, xb, xe, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    // tensor-core kernel: pairs of heads of P = 64 rows, 32-column boxes of both heads' rows, and both
    // heads' logs of x rows as far as the longest window reaches (up to kMaxTmaLog rows)
    if (p.P == 64 && p.H % 2 == 0 && p.hpg % 2 == 0) {
        const cuuint32_t sb2[2] = {32u, 128u};
        const cuuint32_t xb2[3] = {(cuuint32_t)p.P, 2u, (cuuint32_t)p.wwin};
        p.tm_tc_ok = enc(&p.tm_state2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.state, sd, ss, sb2, se,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
                     enc(&p.tm_logx2, xt, 3, p.log_x, xd, xst, xb2, xe, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        // the fold's B operand: logged rows s of group g, [slot * wcap + s][g][n] bf16, boxes of
        // fold_kp rows (the longest window rounded up to a K step multiple: 32, 48 or 64) x 64 columns
        // with the 128-byte swizzle (an MN-major operand tile)
        const int kp = p.wwin <= 32 ? 32 : (p.wwin + 15) / 16 * 16;
        if (p.tm_tc_ok && p.cfg.input_dtype == SSM_DTYPE_BF16 && p.N == 128 && kp <= kMaxFoldK) {
            const cuuint64_t bd[3] = {(cuuint64_t)p.N, (cuuint64_t)p.G, (cuuint64_t)p.n_slots * p.wcap};
            const cuuint64_t bst[2] = {(cuuint64_t)p.N * 2, (cuuint64_t)p.G * p.N * 2};
            const cuuint32_t bb[3] = {64u, 1u, (cuuint32_t)kp};
            p.tm_fold_ok = enc(&p.tm_logB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.log_B, bd, bst, bb, xe,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
            if (p.tm_fold_ok) p.fold_kp = kp;
        }
        // fold in verify: both heads' whole logs (the step is staged after a full log)
        if (p.tm_fold_ok && p.fold_in_verify) {
            const cuuint32_t xbf[3] = {(cuuint32_t)p.P, 2u, (cuuint32_t)p.wcap};
            p.tm_fold_ok = enc(&p.tm_logx_fv, xt, 3, p.log_x, xd, xst, xbf, xe, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
    }
    return p.tm_ok || p.tm_tc_ok;
}

size_t replay_coef_smem_bytes(const Pool &pool, int n_tok) {
    return gcoef_smem_bytes(n_tok, pool.wcap - pool.t1max + n_tok, pool.N, kCoefThreads / 32,
                            (size_t)n_tok * pool.hpg * pool.P * pool.in_bytes, pool.in_bytes, pool.hpg);
}

cudaError_t launch_verify_replay_tma(const Pool &pool, const StepArgs &a, cudaStream_t s, const char **path) {
    if ((!pool.tm_ok && !pool.tm_tc_ok) || !a.wsc || !a.cf || !a.dec) return cudaErrorNotSupported;
    const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
    const int in_b = bf ? 2 : 4;
    if (a.N > 128 || a.wcap > kMaxTmaLog || (a.hpg * a.P * in_b) % 16 || (a.N * in_b) % 16)
        return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(a.x) % 16 || reinterpret_cast<uintptr_t>(a.B) % 16 ||
        reinterpret_cast<uintptr_t>(a.C) % 16)
        return cudaErrorNotSupported;
    const int T1 = a.n_tok;
    const size_t csmem = replay_coef_smem_bytes(pool, T1);
    int dev = 0, max_smem = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (csmem > (size_t)max_smem) return cudaErrorNotSupported;

    // the streaming kernel first, since it fixes the layout the coefficient kernel writes C in:
    // tensor cores take pairs of heads and at most 32 step tokens; W rows are whole float4 (cb_w a
    // multiple of 4, zero past each row's length)
    int NM = 0, nring = 0, naux = 0;
    size_t tsmem = 0;
    if (pool.tm_tc_ok && T1 <= 32 && T1 <= pool.cf_rows && a.P == 64 && a.cb_w % 4 == 0 && a.N <= 128 &&
        (a.N * in_b) % 128 == 0) {
        NM = T1 <= 16 ? 16 : 32;
        if (NM > pool.cf_rows) NM = 0;
        // The ring holds an even number of blocks: the two split groups take alternate blocks, so each
        // slot then belongs to one group, which takes its blocks in order and has seen the slot's
        // previous block land before it waits on the slot again (a parity wait cannot tell a phase two
        // back from the one it waits for).
        static_assert(kTcMaxRing % 2 == 0, "");
        for (int na = kTcMaxAux; NM && na >= 2 && !nring; na -= 2)
            for (int nr = kTcMaxRing; nr >= 4; nr -= 2) {
                const size_t b =
                    tc_smem_bytes(tc_layout(a.N, NM, a.P, in_b, a.wwin, a.t1max, a.cb_w, a.t1pad, !bf, nr, na));
                if (b <= (size_t)max_smem) {
                    nring = nr;
                    naux = na;
                    tsmem = b;
                    break;
                }
            }
    }
    if (!nring && (!pool.tm_ok || a.wcap > 8 * kLogPairs)) return cudaErrorNotSupported;
    const TmaLayout L = tma_layout(a.P, a.N, in_b, T1, a.wcap, a.cb_w);
    // The consumer groups take alternate items, so the stage count is a multiple of the group count:
    // a stage then serves one group, which has consumed the stage's previous item before it waits on
    // the stage again (a parity wait cannot tell a phase two back from the one it waits for).
    static_assert(kMaxStages % kGroups == 0, "");
    const int nstage =
        std::min(kMaxStages, (int)(((long)max_smem - (long)L.fixed) / (long)L.stage)) / kGroups * kGroups;
    if (!nring && nstage < 2) return cudaErrorNotSupported;
    const size_t smem = (size_t)nstage * L.stage + L.fixed;
    StepArgs ac = a;
    ac.cf_nm = nring ? NM : 0;
    if (pool.fold_in_verify && !nring) return cudaErrorNotSupported;

    cudaError_t e = cudaSuccess;
    if (pool.fold_in_verify) {  // the coefficient kernel lists the requests of the two streaming kernels
        e = cudaMemsetAsync(a.counts, 0, 2 * sizeof(int32_t), s);
        if (e != cudaSuccess) return e;
    }
    SSM_DISPATCH_N(a.N, {
        if (bf) {
            auto k = pool.fold_in_verify ? replay_group_coef_kernel<NN, __nv_bfloat16, true>
                                         : replay_group_coef_kernel<NN, __nv_bfloat16, false>;
            e = set_smem(k, csmem);
            if (e != cudaSuccess) return e;
            e = launch_pdl(k, dim3(a.G, a.batch), dim3(kCoefThreads), csmem, s, ac);
        } else {
            auto k = replay_group_coef_kernel<NN, float, false>;
            e = set_smem(k, csmem);
            if (e != cudaSuccess) return e;
            e = launch_pdl(k, dim3(a.G, a.batch), dim3(kCoefThreads), csmem, s, ac);
        }
        if (e != cudaSuccess) return e;
    });
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    if (nring) {
        const int tgrid = std::min(a.batch * (a.H / 2), pool.sm_count);
#define SSM_TC(TI, NMV, LIST)                                                                          \
    do {                                                                                               \
        auto k = verify_replay_tc_kernel<TI, NMV, LIST>;                                               \
        e = set_smem(k, tsmem);                                                                        \
        if (e != cudaSuccess) return e;                                                                \
        cudaLaunchConfig_t cfg = {};                                                                   \
        cudaLaunchAttribute attr[1];                                                                   \
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                               \
        attr[0].val.programmaticStreamSerializationAllowed = 1;                                        \
        cfg.gridDim = dim3(tgrid);                                                                     \
        cfg.blockDim = dim3(TcShape<NMV>::kThreads);                                                   \
        cfg.dynamicSmemBytes = tsmem;                                                                  \
        cfg.stream = s;                                                                                \
        cfg.attrs = attr;                                                                              \
        cfg.numAttrs = 1;                                                                              \
        e = cudaLaunchKernelEx(&cfg, k, ac, pool.tm_state2, pool.tm_logx2, nring, naux);               \
        if (e != cudaSuccess) return e;                                                                \
    } while (0)
        if (bf) {
            if (pool.fold_in_verify) {
                if (NM == 16) SSM_TC(__nv_bfloat16, 16, true);
                else SSM_TC(__nv_bfloat16, 32, true);
            } else {
                if (NM == 16) SSM_TC(__nv_bfloat16, 16, false);
                else SSM_TC(__nv_bfloat16, 32, false);
            }
        } else {
            if (NM == 16) SSM_TC(float, 16, false);
            else SSM_TC(float, 32, false);
        }
#undef SSM_TC
        if (path) *path = "verify_replay_tc";
        if (pool.fold_in_verify) {  // the requests whose full log this verify folds
            e = launch_fold_verify_tc(pool, ac, NM, s);
            if (e != cudaSuccess) return e == cudaErrorNotSupported ? cudaErrorInvalidValue : e;
            if (path) *path = "verify_replay_tc_fold";
        }
        return cudaGetLastError();
    }

    const int n_items = a.batch * a.H;
    const int grid = std::min(n_items, pool.sm_count);
#define SSM_TMA(TI, RP)                                                                                \
    do {                                                                                               \
        auto k = verify_replay_tma_kernel<TI, RP>;                                                     \
        e = set_smem(k, smem);                                                                         \
        if (e != cudaSuccess) return e;                                                                \
        k<<<grid, kTmaThreads, smem, s>>>(ac, pool.tm_state, pool.tm_logx, nstage);                    \
    } while (0)
    if (bf) {
        if (a.P <= 32) SSM_TMA(__nv_bfloat16, 1);
        else SSM_TMA(__nv_bfloat16, 2);
    } else {
        if (a.P <= 32) SSM_TMA(float, 1);
        else SSM_TMA(float, 2);
    }
#undef SSM_TMA
    if (path) *path = "verify_replay_tma";
    return cudaGetLastError();
}

}  // namespace ssm
