// ReplaySSM verify, pipelined (Why Speculative Decoding Slows Hybrid Mamba
// Models, The Fix).  Same arithmetic as verify_replay_kernel in replay.cu:
//
//   y_j[p] = exp(A a_j) (C_j . h_c[p,:]) + sum_{s <= k+j} W[j][s] x_s[p]
//   W[j][s] = exp(A a_{j,s}) dt_s (C_j . B_s)  (+ D for s = k + j)
//
// but organised for the HBM roof: persistent CTAs walk the (request, head)
// items; one producer warp streams each item's checkpoint (32 KiB at
// 64 x 128), its x rows, C rows and C.B rows into a two-stage shared-memory
// ring with bulk copies (TMA), while the consumer warps reduce the previous
// item.  Items are ordered request-major, so the C and C.B rows of a group
// come from L2 after the first head.
//
// Consumer phases per item:
//   A  inclusive prefix sums of dt as fp32 pairs (one warp), then W, decay_j,
//      C in fp32, and the non-finite check of the step inputs;
//   B  the checkpoint rows from shared memory into registers, n_tok FMAs per
//      element for C_j . h_c, xor-shuffle reduction over a row's lanes;
//   C  outputs, and the step's x and dt staged after the log for the commit.
#include "ssm_internal.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kStages = 2;
constexpr int RPT = kRowsPerThread;
constexpr int kPipeMaxThreads = kMaxThreads + 32;  // consumers + one producer warp

__host__ __device__ inline uint32_t up16(uint32_t v) { return (v + 15u) & ~15u; }

// Byte offsets of one stage, and of the unstaged work area after the stages.
struct PipeLayout {
    uint32_t st, xs, cs, cb, dt, hdr, stage;
    uint32_t W, decay, d, Cf, cum, AD, bars, total;
};

__host__ __device__ inline PipeLayout pipe_layout(int P, int N, int in_b, int T1, int mmax, int cb_w, int H) {
    PipeLayout L;
    uint32_t o = 0;
    L.st = o;  o = up16(o + (uint32_t)P * N * 4);
    L.xs = o;  o = up16(o + (uint32_t)mmax * P * in_b);
    L.cs = o;  o = up16(o + (uint32_t)T1 * N * in_b);
    L.cb = o;  o = up16(o + (uint32_t)T1 * cb_w * 4);
    L.dt = o;  o = up16(o + (uint32_t)mmax * 4);
    L.hdr = o; o = up16(o + 16);
    L.stage = (o + 127u) & ~127u;
    o = kStages * L.stage;
    L.W = o;     o = up16(o + (uint32_t)T1 * mmax * 4);
    L.decay = o; o = up16(o + (uint32_t)T1 * 4);
    L.d = o;     o = up16(o + (uint32_t)T1 * P * 4);
    L.Cf = o;    o = up16(o + (uint32_t)T1 * N * 4);
    L.cum = o;   o = up16(o + (uint32_t)mmax * 8);
    L.AD = o;    o = up16(o + (uint32_t)H * 8);
    L.bars = o;  o += 2 * kStages * 8;
    L.total = o;
    return L;
}

__device__ __forceinline__ void raise_flag(uint32_t *flags, uint32_t *slot_flags, int slot, uint32_t bit) {
    atomicOr(flags, bit);
    if (bit != SSM_FLAG_POISONED_SLOT) atomicOr(slot_flags + slot, kSlotPoisoned);
}

// Two consecutive inputs as floats, and two outputs from floats.
__device__ __forceinline__ float2 load2(const float *p) { return *reinterpret_cast<const float2 *>(p); }
__device__ __forceinline__ float2 load2(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
__device__ __forceinline__ void store2(float *p, float a, float b) { *reinterpret_cast<float2 *>(p) = make_float2(a, b); }
__device__ __forceinline__ void store2(__nv_bfloat16 *p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}
__device__ __forceinline__ void copy2(float *d, const float *s) { *reinterpret_cast<float2 *>(d) = *reinterpret_cast<const float2 *>(s); }
__device__ __forceinline__ void copy2(__nv_bfloat16 *d, const __nv_bfloat16 *s) {
    *reinterpret_cast<uint32_t *>(d) = *reinterpret_cast<const uint32_t *>(s);
}

// Barrier over the consumer threads that also ORs a predicate across them.
__device__ __forceinline__ bool consumers_or(int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int N, typename TI>
__global__ void __launch_bounds__(kPipeMaxThreads) verify_replay_pipe_kernel(const __grid_constant__ StepArgs a,
                                                                             int ncw) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    extern __shared__ __align__(128) unsigned char smem[];
    const int P = a.P, T1 = a.n_tok, H = a.H;
    const int wmax = a.wcap - a.t1max;  // W - 1
    const int mmax = wmax + T1;
    const PipeLayout L = pipe_layout(P, N, (int)sizeof(TI), T1, mmax, a.cb_w, H);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kStages;
    float *sAD = reinterpret_cast<float *>(smem + L.AD);  // A[h], D[h] interleaved
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nct = ncw * 32;  // consumer threads
    const int n_items = a.batch * H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], ncw);
        }
        mbar_fence_init();
    }
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        sAD[2 * h] = a.A[h];
        sAD[2 * h + 1] = a.D[h];
    }
    __syncthreads();

    if (warp == ncw) {
        // ------------------------------------------------------------ producer
        const size_t in_b = sizeof(TI);
        // the last item issued to each stage: before the producer leaves, normally or after a wait
        // that ran out, every copy it issued has landed (bounded waits), so none is still writing
        // shared memory when the CTA exits, even if the consumers have already left
        int last[kStages];
        for (int s = 0; s < kStages; ++s) last[s] = -1;
        auto drain = [&]() {
            if (lane == 0)
                for (int s = 0; s < kStages; ++s)
                    if (last[s] >= 0 && !mbar_wait(&full[s], (uint32_t)(last[s] / kStages) & 1u))
                        atomicOr(a.flags, SSM_FLAG_TIMEOUT);
            __syncwarp();
        };
        int n = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
            const int st = n % kStages;
            if (n >= kStages && !mbar_wait(&empty[st], (uint32_t)((n / kStages) - 1) & 1u)) {
                if (lane == 0) atomicOr(a.flags, SSM_FLAG_TIMEOUT);
                drain();
                return;
            }
            last[st] = n;
            const int i = item / H, h = item - i * H;
            const int slot = a.slots[i];
            const int g = h / a.hpg;
            unsigned char *S = smem + (size_t)st * L.stage;
            int gate = 0, k = 0;
            if (lane == 0) {
                k = a.log_len[slot];
                if (a.slot_flags[slot] & kSlotPoisoned) gate = SSM_FLAG_POISONED_SLOT;
                else if (k < 0 || k > wmax) gate = SSM_FLAG_BAD_ACCEPT;
            }
            k = __shfl_sync(0xffffffffu, k, 0);
            gate = __shfl_sync(0xffffffffu, gate, 0);
            int *hdr = reinterpret_cast<int *>(S + L.hdr);
            if (gate) {
                if (lane == 0) {
                    hdr[0] = k;
                    hdr[1] = gate;
                    mbar_arrive_expect_tx(&full[st], 0);
                }
                __syncwarp();
                continue;
            }
            const int m = k + T1;
            const int m4 = (m + 3) & ~3;
            const uint32_t bytes = (uint32_t)((size_t)P * N * 4 + (size_t)m * P * in_b + (size_t)T1 * N * in_b +
                                              (size_t)T1 * m4 * 4);
            const TI *lx = reinterpret_cast<const TI *>(a.log_x);
            const TI *sx = reinterpret_cast<const TI *>(a.x);
            const TI *sC = reinterpret_cast<const TI *>(a.C);
            const int n_copies = 1 + m + 2 * T1;
            for (int c = lane; c < n_copies; c += 32) {
                if (c == 0) {
                    bulk_g2s(S + L.st, a.state + ((size_t)slot * H + h) * (size_t)P * N, (uint32_t)P * N * 4, &full[st]);
                } else if (c < 1 + m) {
                    const int s = c - 1;
                    const TI *src = s < k ? lx + (((size_t)slot * a.wcap + s) * H + h) * P
                                          : sx + (((size_t)i * T1 + (s - k)) * H + h) * P;
                    bulk_g2s(S + L.xs + (size_t)s * P * in_b, src, (uint32_t)(P * in_b), &full[st]);
                } else if (c < 1 + m + T1) {
                    const int j = c - 1 - m;
                    bulk_g2s(S + L.cs + (size_t)j * N * in_b, sC + (((size_t)i * T1 + j) * a.G + g) * N,
                             (uint32_t)(N * in_b), &full[st]);
                } else {
                    const int j = c - 1 - m - T1;
                    bulk_g2s(S + L.cb + (size_t)j * a.cb_w * 4, a.cb + (((size_t)i * a.G + g) * a.t1max + j) * a.cb_w,
                             (uint32_t)m4 * 4, &full[st]);
                }
            }
            float *dts = reinterpret_cast<float *>(S + L.dt);
            for (int s = lane; s < m; s += 32)
                dts[s] = s < k ? a.log_dt[((size_t)slot * a.wcap + s) * H + h]
                               : load_dt(a.dt, ((size_t)i * T1 + (s - k)) * H + h, a.dt_bf16);
            if (lane == 0) {
                hdr[0] = k;
                hdr[1] = 0;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
        }
        drain();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int sub = lane % LPR, rw = lane / LPR;
    float *W = reinterpret_cast<float *>(smem + L.W);
    float *decay = reinterpret_cast<float *>(smem + L.decay);
    float *dsm = reinterpret_cast<float *>(smem + L.d);
    float *Cf = reinterpret_cast<float *>(smem + L.Cf);
    Sum2 *cum = reinterpret_cast<Sum2 *>(smem + L.cum);
    const float rcpP2 = 2.0f / (float)P;
    TI *yout = reinterpret_cast<TI *>(a.y);
    TI *wx = reinterpret_cast<TI *>(a.log_x);
    int n = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
        const int st = n % kStages;
        if (!mbar_wait(&full[st], (uint32_t)(n / kStages) & 1u)) {
            if (threadIdx.x == 0) atomicOr(a.flags, SSM_FLAG_TIMEOUT);
            return;
        }
        const unsigned char *S = smem + (size_t)st * L.stage;
        const int *hdr = reinterpret_cast<const int *>(S + L.hdr);
        const int k = hdr[0], gate = hdr[1];
        const int i = item / H, h = item - i * H;
        const int slot = a.slots[i];
        if (gate) {
            if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, (uint32_t)gate);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            continue;
        }
        const int m = k + T1;
        const float A = sAD[2 * h], D = sAD[2 * h + 1];
        const TI *xs = reinterpret_cast<const TI *>(S + L.xs);
        const TI *Cs = reinterpret_cast<const TI *>(S + L.cs);
        const float *cbs = reinterpret_cast<const float *>(S + L.cb);
        const float *dts = reinterpret_cast<const float *>(S + L.dt);

        // phase A: prefix sums of dt (fp32 pairs, so that differences of them
        // are exact to fp32), W, decay, C in fp32, and the step inputs' finiteness
        if (warp == 0) warp_prefix_sum2(dts, cum, m, lane);
        bool bad = false;  // step x is checked in phase C, where it is read anyway
        for (int e = threadIdx.x; e < T1 * N; e += nct) Cf[e] = to_f(Cs[e]);
        for (int j = threadIdx.x; j < T1; j += nct) bad |= !isfinite(dts[k + j]);
        bar_sync_named(1, nct);  // cum visible
        const float rcpm = 1.0f / (float)m;
        for (int t = threadIdx.x; t < T1 * m; t += nct) {
            const int j = (int)(((float)t + 0.5f) * rcpm), s = t - j * m;
            float w = 0.f;
            if (s <= k + j) {
                const float after = sum2_diff(cum[k + j], cum[s]);
                w = expf(A * after) * dts[s] * cbs[(size_t)j * a.cb_w + s];
                if (s == k + j) w += D;  // skip connection D x_j
            }
            W[t] = w;
        }
        for (int j = threadIdx.x; j < T1; j += nct) decay[j] = expf(A * (cum[k + j].hi + cum[k + j].lo));
        if (consumers_or(nct, bad)) {
            if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            continue;
        }

        // phase B: C_j . h_c[p,:]
        const float4 *st4 = reinterpret_cast<const float4 *>(S + L.st);
        float4 v[RPT][4];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = (warp * RPT + r) * RPW + rw;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[r][q] = p < P ? st4[((size_t)p * N) / 4 + sub + LPR * q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float4 *C4 = reinterpret_cast<const float4 *>(Cf);
        for (int j = 0; j < T1; ++j) {
            float4 c[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) c[q] = C4[(size_t)j * (N / 4) + sub + LPR * q];
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc2 = ffma2(make_float2(c[q].x, c[q].y), make_float2(v[r][q].x, v[r][q].y), acc2);
                    acc2 = ffma2(make_float2(c[q].z, c[q].w), make_float2(v[r][q].z, v[r][q].w), acc2);
                }
                const float acc = row_sum<LPR>(acc2.x + acc2.y);
                const int p = (warp * RPT + r) * RPW + rw;
                if (sub == 0 && p < P) dsm[(size_t)j * P + p] = acc;
            }
        }
        bar_sync_named(1, nct);

        // phase C: outputs (two rows p per thread), the step's x and dt
        // staged after the log, and the non-finite check of the step's x
        const int P2 = P >> 1;
        for (int e = threadIdx.x; e < T1 * P2; e += nct) {
            const int j = (int)(((float)e + 0.5f) * rcpP2), pp = e - j * P2;
            const float dec = decay[j];
            float2 acc = make_float2(dec * dsm[(size_t)j * P + 2 * pp], dec * dsm[(size_t)j * P + 2 * pp + 1]);
            const float *wj = W + (size_t)j * m;
            const int last = k + j;
            for (int s = 0; s <= last; ++s) {
                const float w = wj[s];
                acc = ffma2(make_float2(w, w), load2(xs + (size_t)s * P + 2 * pp), acc);
            }
            const float acc0 = acc.x, acc1 = acc.y;
            const float2 xl = load2(xs + (size_t)last * P + 2 * pp);
            bad |= !isfinite(xl.x) || !isfinite(xl.y);
            store2(yout + (((size_t)i * T1 + j) * H + h) * P + 2 * pp, acc0, acc1);
            copy2(wx + (((size_t)slot * a.wcap + last) * H + h) * P + 2 * pp, xs + (size_t)last * P + 2 * pp);
        }
        for (int j = threadIdx.x; j < T1; j += nct) a.log_dt[((size_t)slot * a.wcap + k + j) * H + h] = dts[k + j];
        if (consumers_or(nct, bad) && threadIdx.x == 0)  // also: the stage and work area are free again
            raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
}

// ---------------------------------------------------------------------------
// Fold, pipelined: the (request, head) pairs listed by the commit walk the
// same kind of ring.  Per item the producer brings the checkpoint and the m
// logged rows of x and B; the consumers form w_s = exp(A sum_{r>s} dt_r) dt_s
// from prefix sums of dt kept as fp32 pairs, then h <- exp(A sum dt) h + sum_s (w_s x_s) (x) B_s
// with m FMAs per element, and store the checkpoint back from registers.

struct FoldLayout {
    uint32_t st, xs, bs, dt, hdr, stage;
    uint32_t xw, bf, cum, sw, A, bars, total;
};

__host__ __device__ inline FoldLayout fold_layout(int P, int N, int in_b, int mmax, int H) {
    FoldLayout L;
    uint32_t o = 0;
    L.st = o;  o = up16(o + (uint32_t)P * N * 4);
    L.xs = o;  o = up16(o + (uint32_t)mmax * P * in_b);
    L.bs = o;  o = up16(o + (uint32_t)mmax * N * in_b);
    L.dt = o;  o = up16(o + (uint32_t)mmax * 4);
    L.hdr = o; o = up16(o + 16);
    L.stage = (o + 127u) & ~127u;
    o = kStages * L.stage;
    L.xw = o;  o = up16(o + (uint32_t)mmax * P * 4);
    L.bf = o;  o = up16(o + (uint32_t)mmax * N * 4);
    L.cum = o; o = up16(o + (uint32_t)mmax * 8);
    L.sw = o;  o = up16(o + (uint32_t)mmax * 4 + 4);  // + the total decay
    L.A = o;   o = up16(o + (uint32_t)H * 4);
    L.bars = o; o += 2 * kStages * 8;
    L.total = o;
    return L;
}

template <int N, typename TI>
__global__ void __launch_bounds__(kPipeMaxThreads) fold_pipe_kernel(const __grid_constant__ CommitArgs a, int ncw) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    extern __shared__ __align__(128) unsigned char smem[];
    const int P = a.P, H = a.H;
    const int mmax = a.wcap;
    const FoldLayout L = fold_layout(P, N, (int)sizeof(TI), mmax, H);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kStages;
    float *sA = reinterpret_cast<float *>(smem + L.A);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nct = ncw * 32;
    const int n_items = *a.fold_count * H;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], ncw);
        }
        mbar_fence_init();
    }
    for (int h = threadIdx.x; h < H; h += blockDim.x) sA[h] = a.A[h];
    __syncthreads();

    if (warp == ncw) {
        // ------------------------------------------------------------ producer
        const size_t in_b = sizeof(TI);
        const TI *lx = reinterpret_cast<const TI *>(a.log_x);
        const TI *lB = reinterpret_cast<const TI *>(a.log_B);
        // as in the verify's producer: every issued copy has landed before the producer leaves
        int last[kStages];
        for (int s = 0; s < kStages; ++s) last[s] = -1;
        auto drain = [&]() {
            if (lane == 0)
                for (int s = 0; s < kStages; ++s)
                    if (last[s] >= 0 && !mbar_wait(&full[s], (uint32_t)(last[s] / kStages) & 1u))
                        atomicOr(a.flags, SSM_FLAG_TIMEOUT);
            __syncwarp();
        };
        int n = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
            const int st = n % kStages;
            if (n >= kStages && !mbar_wait(&empty[st], (uint32_t)((n / kStages) - 1) & 1u)) {
                if (lane == 0) atomicOr(a.flags, SSM_FLAG_TIMEOUT);
                drain();
                return;
            }
            last[st] = n;
            const int f = item / H, h = item - f * H;
            const int2 it = a.fold_items[f];
            const int m = it.y;
            const int slot = a.slots[it.x];
            const int g = h / a.hpg;
            unsigned char *S = smem + (size_t)st * L.stage;
            const uint32_t bytes = (uint32_t)((size_t)P * N * 4 + (size_t)m * (P + N) * in_b);
            for (int c = lane; c < 1 + 2 * m; c += 32) {
                if (c == 0) {
                    bulk_g2s(S + L.st, a.state + ((size_t)slot * H + h) * (size_t)P * N, (uint32_t)P * N * 4, &full[st]);
                } else if (c <= m) {
                    const int s = c - 1;
                    bulk_g2s(S + L.xs + (size_t)s * P * in_b, lx + (((size_t)slot * a.wcap + s) * H + h) * P,
                             (uint32_t)(P * in_b), &full[st]);
                } else {
                    const int s = c - 1 - m;
                    bulk_g2s(S + L.bs + (size_t)s * N * in_b, lB + (((size_t)slot * a.wcap + s) * a.G + g) * N,
                             (uint32_t)(N * in_b), &full[st]);
                }
            }
            float *dts = reinterpret_cast<float *>(S + L.dt);
            for (int s = lane; s < m; s += 32) dts[s] = a.log_dt[((size_t)slot * a.wcap + s) * H + h];
            if (lane == 0) {
                int *hdr = reinterpret_cast<int *>(S + L.hdr);
                hdr[0] = m;
                hdr[1] = slot;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
        }
        drain();
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int sub = lane % LPR, rw = lane / LPR;
    float *xw = reinterpret_cast<float *>(smem + L.xw);
    float *bf = reinterpret_cast<float *>(smem + L.bf);
    Sum2 *cum = reinterpret_cast<Sum2 *>(smem + L.cum);
    float *sw = reinterpret_cast<float *>(smem + L.sw);
    const float rcpP = 1.0f / (float)P;
    int n = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++n) {
        const int st = n % kStages;
        if (!mbar_wait(&full[st], (uint32_t)(n / kStages) & 1u)) {
            if (threadIdx.x == 0) atomicOr(a.flags, SSM_FLAG_TIMEOUT);
            return;
        }
        const unsigned char *S = smem + (size_t)st * L.stage;
        const int *hdr = reinterpret_cast<const int *>(S + L.hdr);
        const int m = hdr[0], slot = hdr[1];
        const int h = item - (item / H) * H;
        const float A = sA[h];
        const TI *xs = reinterpret_cast<const TI *>(S + L.xs);
        const TI *bs = reinterpret_cast<const TI *>(S + L.bs);
        const float *dts = reinterpret_cast<const float *>(S + L.dt);

        if (warp == 0) warp_prefix_sum2(dts, cum, m, lane);  // differences exact to fp32
        for (int e = threadIdx.x; e < m * N; e += nct) bf[e] = to_f(bs[e]);
        bar_sync_named(1, nct);
        for (int s = threadIdx.x; s < m; s += nct)  // exp(A * dt applied after token s) dt_s
            sw[s] = expf(A * sum2_diff(cum[m - 1], cum[s])) * dts[s];
        if (threadIdx.x == 0) sw[mmax] = expf(A * (cum[m - 1].hi + cum[m - 1].lo));
        bar_sync_named(1, nct);
        for (int e = threadIdx.x; e < m * P; e += nct) {
            const int s = (int)(((float)e + 0.5f) * rcpP);
            xw[e] = sw[s] * to_f(xs[e]);
        }
        bar_sync_named(1, nct);

        const float decay = sw[mmax];
        const float4 *st4 = reinterpret_cast<const float4 *>(S + L.st);
        const float4 *B4 = reinterpret_cast<const float4 *>(bf);
        float *gst = a.state + ((size_t)slot * H + h) * (size_t)P * N;
        int prow[RPT];
        float2 v[RPT][8];  // the thread's 16 values of each of its rows, as pairs
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = (warp * RPT + r) * RPW + rw;
            prow[r] = p < P ? p : 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 f = st4[((size_t)prow[r] * N) / 4 + sub + LPR * q];
                v[r][2 * q] = make_float2(f.x * decay, f.y * decay);
                v[r][2 * q + 1] = make_float2(f.z * decay, f.w * decay);
            }
        }
        for (int s = 0; s < m; ++s) {
            float4 b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) b[q] = B4[(size_t)s * (N / 4) + sub + LPR * q];
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float u = xw[(size_t)s * P + prow[r]];
                const float2 uu = make_float2(u, u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[r][2 * q] = ffma2(uu, make_float2(b[q].x, b[q].y), v[r][2 * q]);
                    v[r][2 * q + 1] = ffma2(uu, make_float2(b[q].z, b[q].w), v[r][2 * q + 1]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = (warp * RPT + r) * RPW + rw;
            if (p < P)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_stream(gst + (size_t)p * N + 4 * (sub + LPR * q),
                              make_float4(v[r][2 * q].x, v[r][2 * q].y, v[r][2 * q + 1].x, v[r][2 * q + 1].y));
        }
        bar_sync_named(1, nct);  // the stage and the work area are free again
        if (lane == 0) mbar_arrive(&empty[st]);
    }
}

}  // namespace

cudaError_t launch_verify_replay_pipe(const Pool &pool, const StepArgs &a, cudaStream_t s) {
    const int in_b = pool.cfg.input_dtype == SSM_DTYPE_BF16 ? 2 : 4;
    // bulk copies move 16-byte multiples between 16-byte aligned addresses
    if ((a.P * in_b) % 16 || (a.N * in_b) % 16 || a.cb_w % 4) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(a.x) % 16 || reinterpret_cast<uintptr_t>(a.C) % 16 ||
        reinterpret_cast<uintptr_t>(a.log_x) % 16 || reinterpret_cast<uintptr_t>(a.cb) % 16 ||
        reinterpret_cast<uintptr_t>(a.state) % 16)
        return cudaErrorNotSupported;
    const int rows = (32 / (a.N / 16)) * RPT;
    const int ncw = (a.P + rows - 1) / rows;
    if (32 * ncw > kMaxThreads) return cudaErrorNotSupported;
    const int mmax = a.wcap - a.t1max + a.n_tok;
    const PipeLayout L = pipe_layout(a.P, a.N, in_b, a.n_tok, mmax, a.cb_w, a.H);
    int dev = 0, max_smem = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (L.total > (uint32_t)max_smem) return cudaErrorNotSupported;
    const int per_sm = (int)(2 * L.total) <= max_smem ? 2 : 1;
    const int items = a.batch * a.H;
    const int grid = items < per_sm * pool.sm_count ? items : per_sm * pool.sm_count;
    const bool bf = in_b == 2;
    SSM_DISPATCH_N(a.N, {
        const dim3 block(32 * (ncw + 1));
        if (bf) {
            auto k = verify_replay_pipe_kernel<NN, __nv_bfloat16>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
            if (e != cudaSuccess) return e;
            k<<<grid, block, L.total, s>>>(a, ncw);
        } else {
            auto k = verify_replay_pipe_kernel<NN, float>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
            if (e != cudaSuccess) return e;
            k<<<grid, block, L.total, s>>>(a, ncw);
        }
    });
    return cudaGetLastError();
}

}  // namespace ssm

namespace ssm {

cudaError_t launch_fold_pipe(const Pool &pool, const CommitArgs &a, cudaStream_t s) {
    const int in_b = pool.cfg.input_dtype == SSM_DTYPE_BF16 ? 2 : 4;
    if ((a.P * in_b) % 16 || (a.N * in_b) % 16) return cudaErrorNotSupported;
    if (reinterpret_cast<uintptr_t>(a.log_x) % 16 || reinterpret_cast<uintptr_t>(a.log_B) % 16 ||
        reinterpret_cast<uintptr_t>(a.state) % 16)
        return cudaErrorNotSupported;
    const int rows = (32 / (a.N / 16)) * RPT;
    const int ncw = (a.P + rows - 1) / rows;
    if (32 * ncw > kMaxThreads) return cudaErrorNotSupported;
    const FoldLayout L = fold_layout(a.P, a.N, in_b, a.wcap, a.H);
    int dev = 0, max_smem = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (L.total > (uint32_t)max_smem) return cudaErrorNotSupported;
    const int per_sm = (int)(2 * L.total) <= max_smem ? 2 : 1;
    const int grid = per_sm * pool.sm_count;
    const bool bf = in_b == 2;
    SSM_DISPATCH_N(a.N, {
        const dim3 block(32 * (ncw + 1));
        if (bf) {
            auto k = fold_pipe_kernel<NN, __nv_bfloat16>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
            if (e != cudaSuccess) return e;
            k<<<grid, block, L.total, s>>>(a, ncw);
        } else {
            auto k = fold_pipe_kernel<NN, float>;
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
            if (e != cudaSuccess) return e;
            k<<<grid, block, L.total, s>>>(a, ncw);
        }
    });
    return cudaGetLastError();
}

}  // namespace ssm
