// ReplaySSM verify, and the commit of a verify step (copy and replay pools).
//
// Replay verify (Why Speculative Decoding Slows Hybrid Mamba Models, The
// Fix): with the checkpoint h_c, the k logged tokens and the step tokens
// u_k .. u_{k+n_tok-1} forming one token sequence u, the output of step
// token j (m = k + j + 1 tokens applied) is
//
//   y_j[p] = exp(A a_j) (C_j . h_c[p,:]) + sum_{s<m} W[j][s] x_s[p]
//   W[j][s] = exp(A a_{j,s}) dt_s (C_j . B_s)  (+ D for s = m - 1, the skip term)
//
// where a_j is the sum of all m applied dt and a_{j,s} the sum of the dt
// applied after token s.  Two kernels:
//   replay_prep   one CTA per (request, group): C_j . B_s for the pairs
//                 s <= k + j, into pool scratch (shared by the group's heads);
//                 also appends the step's B after the log;
//   verify_replay one CTA per (request, head): reads the checkpoint once,
//                 n_tok FMAs per state element for C_j . h_c, then the small
//                 W X product from shared memory.  No state is written.
//
// The commit (same page, The Fix; The Problem for the copy flavour): a
// one-thread-per-request kernel makes the index decisions (bit exact): copy
// pools move the slot's current-state index onto the snapshot of the last
// kept token; replay pools append the kept tokens (already staged after the
// log) or, when the window would fill, list the request for a fold.  A
// persistent kernel then folds only the listed (request, head) pairs in
// closed form, h <- exp(A a) h + sum_s (exp(A a_s) dt_s x_s) (x) B_s.
#include <cstring>
#include <mutex>

#include "pdl.cuh"
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int RPT = kRowsPerThread;

template <int N>
int warps_for(int P) {
    const int rows = (32 / (N / 16)) * RPT;
    return (P + rows - 1) / rows;
}

__device__ __forceinline__ void raise_flag(uint32_t *flags, uint32_t *slot_flags, int slot, uint32_t bit) {
    atomicOr(flags, bit);
    if (bit != SSM_FLAG_POISONED_SLOT) atomicOr(slot_flags + slot, kSlotPoisoned);
}

__device__ __forceinline__ size_t cb_index(const StepArgs &a, int i, int g, int j, int s) {
    return (((size_t)i * a.G + g) * a.t1max + j) * a.cb_w + s;
}

// ------------------------------------------------------------------ prep: C_j . B_s per group

template <int N, typename TI>
__global__ void __launch_bounds__(256) replay_prep_kernel(const __grid_constant__ StepArgs a) {
    extern __shared__ float4 smem4[];
    const int g = blockIdx.x, i = blockIdx.y;
    const int slot = a.slots[i];
    const int T1 = a.n_tok;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int wmax = a.wcap - a.t1max;
    const int k = a.log_len[slot];
    if ((a.slot_flags[slot] & kSlotPoisoned) || k < 0 || k > wmax) return;  // the main kernel reports it
    const int m = k + T1;
    float *sC = reinterpret_cast<float *>(smem4);  // [T1][N]
    float *sB = sC + (size_t)T1 * N;               // [m][N]
    const TI *lB = reinterpret_cast<const TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    TI *wB = reinterpret_cast<TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    const TI *stepB = reinterpret_cast<const TI *>(a.B);
    const TI *stepC = reinterpret_cast<const TI *>(a.C);
    bool bad = false;
    for (int e = threadIdx.x; e < T1 * N; e += blockDim.x) {
        const int j = e / N, n = e - j * N;
        const float c = to_f(stepC[(((size_t)i * T1 + j) * a.G + g) * N + n]);
        bad |= !isfinite(c);
        sC[e] = c;
    }
    for (int e = threadIdx.x; e < m * N; e += blockDim.x) {
        const int s = e / N, n = e - s * N;
        float b;
        if (s < k) {
            b = to_f(lB[((size_t)s * a.G + g) * N + n]);
        } else {
            const TI raw = stepB[(((size_t)i * T1 + (s - k)) * a.G + g) * N + n];
            b = to_f(raw);
            bad |= !isfinite(b);
            wB[((size_t)s * a.G + g) * N + n] = raw;  // staged after the log for the commit
        }
        sB[e] = b;
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }
    // one warp per (j, s) pair with s <= k + j, lanes over n
    for (int pr = warp; pr < T1 * m; pr += nwarps) {
        const int j = pr / m, s = pr - j * m;
        if (s > k + j) continue;
        float dot = 0.f;
#pragma unroll
        for (int n = lane; n < N; n += 32) dot = fmaf(sC[(size_t)j * N + n], sB[(size_t)s * N + n], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) a.cb[cb_index(a, i, g, j, s)] = dot;
    }
}

// ------------------------------------------------------------------ verify

struct ReplaySmem {
    float *C, *x, *dt, *W, *decay, *d;
};

// C first: N is a multiple of 16, so C stays 16-byte aligned for float4 reads.
__host__ __device__ inline size_t replay_floats(int m, int n_tok, int N, int P) {
    return (size_t)n_tok * N + (size_t)m * P + m + (size_t)n_tok * m + n_tok + (size_t)n_tok * P;
}

__device__ inline ReplaySmem carve(float *base, int m, int n_tok, int N, int P) {
    ReplaySmem s;
    s.C = base;
    s.x = s.C + (size_t)n_tok * N;
    s.dt = s.x + (size_t)m * P;
    s.W = s.dt + m;
    s.decay = s.W + (size_t)n_tok * m;
    s.d = s.decay + n_tok;
    return s;
}

template <int N, typename TI>
__global__ void __launch_bounds__(kMaxThreads) verify_replay_kernel(const __grid_constant__ StepArgs a) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    extern __shared__ float4 smem4[];
    __shared__ uint32_t s_gate;
    __shared__ int s_k;
    const int h = blockIdx.x, i = blockIdx.y;
    const int slot = a.slots[i];
    const int g = h / a.hpg;
    const int P = a.P, T1 = a.n_tok;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, rw = lane / LPR;
    const int wmax = a.wcap - a.t1max;  // W - 1, the largest legal log length

    if (threadIdx.x == 0) {
        const int k = a.log_len[slot];
        uint32_t gate = 0;
        if (a.slot_flags[slot] & kSlotPoisoned) gate = SSM_FLAG_POISONED_SLOT;
        else if (k < 0 || k > wmax) gate = SSM_FLAG_BAD_ACCEPT;  // corrupted log length
        s_gate = gate;
        s_k = k;
    }

    // checkpoint rows: the only large read of this kernel
    const float *hc = a.state + ((size_t)slot * a.H + h) * (size_t)P * N;
    float4 v[RPT][4];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int p = (warp * RPT + r) * RPW + rw;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            v[r][q] = p < P ? ld_stream(hc + (size_t)p * N + 4 * (sub + LPR * q)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    if (s_gate) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, s_gate);
        return;
    }
    const int k = s_k;
    const int m = k + T1;
    ReplaySmem sm = carve(reinterpret_cast<float *>(smem4), m, T1, N, P);
    const float A = a.A[h], D = a.D[h];

    const TI *lx = reinterpret_cast<const TI *>(a.log_x) + (size_t)slot * a.wcap * a.H * P;
    const float *ldt = a.log_dt + (size_t)slot * a.wcap * a.H;
    TI *wx = reinterpret_cast<TI *>(a.log_x) + (size_t)slot * a.wcap * a.H * P;
    float *wdt = a.log_dt + (size_t)slot * a.wcap * a.H;
    const TI *sx = reinterpret_cast<const TI *>(a.x);
    const TI *sC = reinterpret_cast<const TI *>(a.C);

    // x and dt of the token sequence u = log[0..k) ++ step tokens; the step's
    // x and dt are staged after the log for the commit.  C was checked by
    // the prep kernel (which poisons the slot before this kernel runs).
    bool bad = false;
    for (int e = threadIdx.x; e < m * P; e += blockDim.x) {
        const int s = e / P, p = e - s * P;
        float xv;
        if (s < k) {
            xv = to_f(lx[((size_t)s * a.H + h) * P + p]);
        } else {
            const TI raw = sx[(((size_t)i * T1 + (s - k)) * a.H + h) * P + p];
            xv = to_f(raw);
            bad |= !isfinite(xv);
            wx[((size_t)s * a.H + h) * P + p] = raw;
        }
        sm.x[e] = xv;
    }
    for (int s = threadIdx.x; s < m; s += blockDim.x) {
        float d;
        if (s < k) {
            d = ldt[(size_t)s * a.H + h];
        } else {
            d = load_dt(a.dt, ((size_t)i * T1 + (s - k)) * a.H + h, a.dt_bf16);
            bad |= !isfinite(d);
            wdt[(size_t)s * a.H + h] = d;
        }
        sm.dt[s] = d;
    }
    for (int e = threadIdx.x; e < T1 * N; e += blockDim.x) {
        const int j = e / N, n = e - j * N;
        sm.C[e] = to_f(sC[(((size_t)i * T1 + j) * a.G + g) * N + n]);
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }

    // W[j][s]: one thread per pair; the dt applied after token s are summed
    // newest first (the time elapsed since token s)
    for (int t = threadIdx.x; t < T1 * m; t += blockDim.x) {
        const int j = t / m, s = t - j * m;
        float w = 0.f;
        if (s <= k + j) {
            float after = 0.f;
            for (int r = k + j; r > s; --r) after += sm.dt[r];
            w = expf(A * after) * sm.dt[s] * a.cb[cb_index(a, i, g, j, s)];
            if (s == k + j) w += D;  // skip connection D x_j
        }
        sm.W[t] = w;
    }
    for (int j = threadIdx.x; j < T1; j += blockDim.x) {
        float total = 0.f;
        for (int r = k + j; r >= 0; --r) total += sm.dt[r];
        sm.decay[j] = expf(A * total);
    }

    // C_j . h_c[p,:] for every step token and row
    const float4 *C4 = reinterpret_cast<const float4 *>(sm.C);
    for (int j = 0; j < T1; ++j) {
        float4 c[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) c[q] = C4[(size_t)j * (N / 4) + sub + LPR * q];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc = fmaf(c[q].x, v[r][q].x, acc);
                acc = fmaf(c[q].y, v[r][q].y, acc);
                acc = fmaf(c[q].z, v[r][q].z, acc);
                acc = fmaf(c[q].w, v[r][q].w, acc);
            }
            acc = row_sum<LPR>(acc);
            const int p = (warp * RPT + r) * RPW + rw;
            if (sub == 0 && p < P) sm.d[(size_t)j * P + p] = acc;
        }
    }
    __syncthreads();

    // y_j[p] = decay_j d_j[p] + sum_{s <= k+j} W[j][s] x_s[p]
    TI *y = reinterpret_cast<TI *>(a.y);
    for (int e = threadIdx.x; e < T1 * P; e += blockDim.x) {
        const int j = e / P, p = e - j * P;
        float acc = sm.decay[j] * sm.d[e];
        const float *wj = sm.W + (size_t)j * m;
        for (int s = 0; s <= k + j; ++s) acc = fmaf(wj[s], sm.x[(size_t)s * P + p], acc);
        y[(((size_t)i * T1 + j) * a.H + h) * P + p] = from_f<TI>(acc);
    }
}

// ------------------------------------------------------------------ commit

// Decision of one request: tokens committed (c) and whether the log is
// folded.  Returns false when the request is skipped (err says why).
__device__ __forceinline__ bool commit_decision(const CommitArgs &a, int i, int slot, int k, int &c, bool &fold,
                                                uint32_t &err) {
    err = 0;
    if (a.slot_flags[slot] & kSlotPoisoned) { err = SSM_FLAG_POISONED_SLOT; return false; }
    if (a.flush) {
        c = 0;
        fold = k > 0;
        return true;
    }
    const int acc = a.accept[i];
    if (acc < 0 || acc >= a.ntok[i]) { err = SSM_FLAG_BAD_ACCEPT; return false; }
    c = acc + 1;
    fold = a.force_fold || (k + c >= a.W);
    return true;
}

// Fold in verify: the kept tokens' log rows of one slot move from row `from`
// to row `to` (to < from): x, B and dt rows each form one contiguous range.
// Disjoint ranges are copied in kMoveParts slices by as many CTAs; ranges
// that overlap (from < to + c, possible when W < the step's tokens) are
// copied by one CTA row by row in increasing order, a barrier between rows,
// so that every source row is read before it is overwritten.
constexpr int kMoveParts = 8;
constexpr int kMoveThreads = 256;

template <typename V>
__device__ void move_range(char *base, size_t row_bytes, int from, int to, int c, bool overlap) {
    const V *src = reinterpret_cast<const V *>(base + (size_t)from * row_bytes);
    V *dst = reinterpret_cast<V *>(base + (size_t)to * row_bytes);
    const size_t rw = row_bytes / sizeof(V);
    if (!overlap) {
        const size_t n = rw * (size_t)c, per = (n + kMoveParts - 1) / kMoveParts;
        const size_t e0 = per * blockIdx.y, e1 = min(n, e0 + per);
        for (size_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) dst[e] = src[e];
        return;
    }
    if (blockIdx.y != 0) return;
    for (int r = 0; r < c; ++r) {
        for (size_t e = threadIdx.x; e < rw; e += blockDim.x) dst[(size_t)r * rw + e] = src[(size_t)r * rw + e];
        __syncthreads();
    }
}

// CTA (listed move, slice).  Launched programmatically after the commit's index kernel: the next verify's
// coefficient kernel may be scheduled as this grid drains (it waits for it); the list is read once the
// index kernel has completed.
__global__ void __launch_bounds__(kMoveThreads) log_move_kernel(const __grid_constant__ CommitArgs a) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if ((int)blockIdx.x >= a.counts[2]) return;
    const int4 mv = a.moves[blockIdx.x];
    const int slot = a.slots[mv.x], from = mv.y, to = mv.z, c = mv.w;
    const bool overlap = from < to + c;
    const size_t xrow = (size_t)a.H * a.P * 2, brow = (size_t)a.G * a.N * 2, drow = (size_t)a.H * 4;  // bf16 x, B
    move_range<uint4>(static_cast<char *>(a.log_x) + (size_t)slot * a.wcap * xrow, xrow, from, to, c, overlap);
    move_range<uint4>(static_cast<char *>(a.log_B) + (size_t)slot * a.wcap * brow, brow, from, to, c, overlap);
    move_range<float>(reinterpret_cast<char *>(a.log_dt) + (size_t)slot * a.wcap * drow, drow, from, to, c,
                      overlap);
}

// One thread per request: the index side of the commit (bit exact).  kMoves:
// a commit of a pool that folds in its verify (appends, moving staged tokens).
// reset: one CTA covers the batch and clears the fold and move counts itself
// (else the host clears them before the launch).
template <bool kMoves>
__global__ void commit_meta_kernel(const __grid_constant__ CommitArgs a, int replay, int reset) {
    // the log move (or the fold) may be scheduled now: it waits for this grid before it reads the lists
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (reset) {
        if (threadIdx.x == 0 && replay) {
            *a.fold_count = 0;
            if (kMoves) a.counts[2] = 0;
        }
        __syncthreads();
    }
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.batch) return;
    const int slot = a.slots[i];
    const int k = replay ? a.log_len[slot] : 0;
    int c = 0;
    bool fold = false;
    uint32_t err = 0;
    if (!commit_decision(a, i, slot, k, c, fold, err)) {
        raise_flag(a.flags, a.slot_flags, slot, err);
        return;
    }
    if (replay) {
        if (k < 0 || k + c > a.wcap) {  // corrupted log length
            raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_BAD_ACCEPT);
            return;
        }
        if constexpr (kMoves) {
            // fold in verify: the window fills in the next verify, and this commit appends; the
            // verify staged its tokens after the log as it then was, and where that log has since
            // gone into the checkpoint (folded by the verify or a checkpoint read) the kept tokens
            // move to the end of the log first
            const int sp = a.stage_pos[slot];
            if (sp != k) {
                if (sp < 0 || sp + c > a.wcap) {
                    raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_BAD_ACCEPT);
                    return;
                }
                a.moves[atomicAdd(&a.counts[2], 1)] = make_int4(i, sp, k, c);
            }
            fold = a.force_fold != 0;
        }
        if (fold) a.fold_items[atomicAdd(a.fold_count, 1)] = make_int2(i, k + c);
        a.log_len[slot] = fold ? 0 : k + c;
    } else {
        const int cur = a.cur[slot];
        const int half = (cur >= 0 && cur < a.t1max) ? 1 : 0;  // the half the verify wrote
        a.cur[slot] = half * a.t1max + (c - 1);
    }
    a.position[slot] += c;
}

// Persistent: CTAs walk the listed (request, head) pairs.
template <int N, typename TI>
__global__ void __launch_bounds__(kMaxThreads) fold_kernel(const __grid_constant__ CommitArgs a) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    extern __shared__ float4 smem4[];
    __shared__ float s_decay;
    const int P = a.P;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, rw = lane / LPR;
    const int total = *a.fold_count * a.H;
    float *sB = reinterpret_cast<float *>(smem4);   // [m][N]

    for (int w = blockIdx.x; w < total; w += gridDim.x) {
        const int2 item = a.fold_items[w / a.H];
        const int h = w - (w / a.H) * a.H;
        const int i = item.x, m = item.y;
        const int slot = a.slots[i];
        const int g = h / a.hpg;
        float *sxw = sB + (size_t)m * N;             // [m][P]  w_s x_s[p]
        float *sdt = sxw + (size_t)m * P;            // [m]
        float *sw = sdt + m;                         // [m]

        float *st = a.state + ((size_t)slot * a.H + h) * (size_t)P * N;
        float4 v[RPT][4];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = (warp * RPT + r) * RPW + rw;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[r][q] = p < P ? ld_stream(st + (size_t)p * N + 4 * (sub + LPR * q)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float A = a.A[h];
        const TI *lx = reinterpret_cast<const TI *>(a.log_x) + (size_t)slot * a.wcap * a.H * P;
        const TI *lB = reinterpret_cast<const TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
        const float *ldt = a.log_dt + (size_t)slot * a.wcap * a.H;
        for (int s = threadIdx.x; s < m; s += blockDim.x) sdt[s] = ldt[(size_t)s * a.H + h];
        for (int e = threadIdx.x; e < m * N; e += blockDim.x) {
            const int s = e / N, n = e - s * N;
            sB[e] = to_f(lB[((size_t)s * a.G + g) * N + n]);
        }
        __syncthreads();
        // decay weight of token s: exp(A * dt applied after it), newest first
        for (int s = threadIdx.x; s < m; s += blockDim.x) {
            float after = 0.f;
            for (int r = m - 1; r > s; --r) after += sdt[r];
            sw[s] = expf(A * after) * sdt[s];
        }
        if (threadIdx.x == 0) {
            float all = 0.f;
            for (int r = m - 1; r >= 0; --r) all += sdt[r];
            s_decay = expf(A * all);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < m * P; e += blockDim.x) {
            const int s = e / P, p = e - s * P;
            sxw[e] = sw[s] * to_f(lx[((size_t)s * a.H + h) * P + p]);
        }
        __syncthreads();

        const float decay = s_decay;
#pragma unroll
        for (int r = 0; r < RPT; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[r][q].x *= decay; v[r][q].y *= decay; v[r][q].z *= decay; v[r][q].w *= decay;
            }
        const float4 *B4 = reinterpret_cast<const float4 *>(sB);
        int prow[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = (warp * RPT + r) * RPW + rw;
            prow[r] = p < P ? p : 0;
        }
        for (int s = 0; s < m; ++s) {
            float4 b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) b[q] = B4[(size_t)s * (N / 4) + sub + LPR * q];
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const float u = sxw[(size_t)s * P + prow[r]];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    v[r][q].x = fmaf(u, b[q].x, v[r][q].x);
                    v[r][q].y = fmaf(u, b[q].y, v[r][q].y);
                    v[r][q].z = fmaf(u, b[q].z, v[r][q].z);
                    v[r][q].w = fmaf(u, b[q].w, v[r][q].w);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int p = (warp * RPT + r) * RPW + rw;
            if (p < P)
#pragma unroll
                for (int q = 0; q < 4; ++q) st_stream(st + (size_t)p * N + 4 * (sub + LPR * q), v[r][q]);
        }
        __syncthreads();  // shared memory is reused by the next item
    }
}

}  // namespace

size_t replay_smem_bytes(const Pool &pool, int n_tok) {
    const int m = pool.wcap - pool.t1max + n_tok;  // W - 1 + n_tok
    return replay_floats(m, n_tok, pool.N, pool.P) * sizeof(float);
}

size_t replay_prep_smem_bytes(const Pool &pool, int n_tok) {
    const int m = pool.wcap - pool.t1max + n_tok;
    return ((size_t)n_tok * pool.N + (size_t)m * pool.N) * sizeof(float);
}

size_t fold_smem_bytes(const Pool &pool) {
    const int m = pool.wcap;
    return ((size_t)m * pool.N + (size_t)m * pool.P + 2 * (size_t)m) * sizeof(float);
}

template <typename K>
static cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_verify_replay(const Pool &pool, const StepArgs &a, cudaStream_t s, const char **path) {
    {  // the tensor-map path brings its own C . B and staging
        const cudaError_t e = launch_verify_replay_tma(pool, a, s, path);
        if (e != cudaErrorNotSupported) return e;
        if (pool.fold_in_verify) return cudaErrorInvalidValue;  // no other path folds in the verify
    }
    const size_t smem = replay_smem_bytes(pool, a.n_tok);
    const size_t psmem = replay_prep_smem_bytes(pool, a.n_tok);
    const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
    SSM_DISPATCH_N(a.N, {
        const dim3 block(32 * warps_for<NN>(a.P));
        if (bf) {
            auto kp = replay_prep_kernel<NN, __nv_bfloat16>;
            cudaError_t e = set_smem(kp, psmem);
            if (e != cudaSuccess) return e;
            kp<<<dim3(a.G, a.batch), 256, psmem, s>>>(a);
        } else {
            auto kp = replay_prep_kernel<NN, float>;
            cudaError_t e = set_smem(kp, psmem);
            if (e != cudaSuccess) return e;
            kp<<<dim3(a.G, a.batch), 256, psmem, s>>>(a);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = launch_verify_replay_pipe(pool, a, s);
        if (e != cudaErrorNotSupported) {
            if (path) *path = "verify_replay_pipe";
            return e;
        }
        if (path) *path = "verify_replay";
        if (bf) {
            auto k = verify_replay_kernel<NN, __nv_bfloat16>;
            e = set_smem(k, smem);
            if (e != cudaSuccess) return e;
            k<<<dim3(a.H, a.batch), block, smem, s>>>(a);
        } else {
            auto k = verify_replay_kernel<NN, float>;
            e = set_smem(k, smem);
            if (e != cudaSuccess) return e;
            k<<<dim3(a.H, a.batch), block, smem, s>>>(a);
        }
    });
    return cudaGetLastError();
}

cudaError_t launch_commit(const Pool &pool, const CommitArgs &a, cudaStream_t s, const char **path) {
    const bool replay = pool.cfg.mode == SSM_MODE_REPLAY;
    const bool moves = a.fold_w && !a.flush;
    // up to 1024 requests one CTA clears the counts in the kernel; else the host clears them first
    const bool one = a.batch <= 1024;
    if (replay && !one) {
        cudaError_t e = cudaMemsetAsync(a.fold_count, 0, sizeof(int32_t), s);
        if (e == cudaSuccess && moves) e = cudaMemsetAsync(&a.counts[2], 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return e;
    }
    const dim3 mgrid(one ? 1u : (unsigned)((a.batch + 127) / 128));
    const dim3 mblock(one ? (unsigned)((a.batch + 31) / 32 * 32) : 128u);
    if (moves) commit_meta_kernel<true><<<mgrid, mblock, 0, s>>>(a, 1, one ? 1 : 0);
    else commit_meta_kernel<false><<<mgrid, mblock, 0, s>>>(a, replay ? 1 : 0, one ? 1 : 0);
    if (path) *path = "commit_copy";
    if (replay) {
        cudaError_t ep = cudaGetLastError();
        if (ep != cudaSuccess) return ep;
        if (moves) {
            ep = launch_pdl(log_move_kernel, dim3(a.batch, kMoveParts), dim3(kMoveThreads), 0, s, a);
            if (ep == cudaSuccess) ep = cudaGetLastError();
            if (ep != cudaSuccess) return ep;
            if (path) *path = "commit_replay_append";
            if (!a.force_fold) return cudaSuccess;  // nothing folds here
        }
        ep = launch_fold_tc(pool, a, s);
        if (path) *path = "commit_replay_fold_tc";
        if (ep != cudaErrorNotSupported) return ep;
        ep = launch_fold_pipe(pool, a, s);
        if (path) *path = "commit_replay_fold_pipe";
        if (ep != cudaErrorNotSupported) return ep;
        if (path) *path = "commit_replay_fold";
        const size_t smem = fold_smem_bytes(pool);
        const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
        SSM_DISPATCH_N(a.N, {
            const dim3 block(32 * warps_for<NN>(a.P));
            if (bf) {
                auto k = fold_kernel<NN, __nv_bfloat16>;
                cudaError_t e = set_smem(k, smem);
                if (e != cudaSuccess) return e;
                k<<<a.fold_grid, block, smem, s>>>(a);
            } else {
                auto k = fold_kernel<NN, float>;
                cudaError_t e = set_smem(k, smem);
                if (e != cudaSuccess) return e;
                k<<<a.fold_grid, block, smem, s>>>(a);
            }
        });
    }
    return cudaGetLastError();
}

}  // namespace ssm

// ---------------------------------------------------------------------------
// Replay verify for callers that cannot allocate device memory.
//
// Code that cannot call cudaMalloc -- a serving engine whose caching
// allocator owns all device memory, or a plugin that is handed only the
// buffers its host runtime manages -- cannot create a pool.  ssm_verify_replay_static runs the same two kernels as
// ssm_verify_replay on buffers the caller owns and takes its scratch (the
// C_j . B_s pair matrix and one status word per request) from the
// file-scope array below, which is part of the library image: every GPU
// that loads the library holds its 4 MiB until the process exits, and no
// call allocates anything.  Every call shares the array, so calls that
// overlap on the GPU (two streams, or two threads) race on it.
namespace ssm {
namespace {

constexpr size_t kStaticScratchFloats = size_t(1) << 20;  // 4 MiB
constexpr size_t kStaticFlagWords = kMaxSlotsPerLaunch;    // per-request status words, at the end
static_assert(kStaticFlagWords < kStaticScratchFloats, "scratch layout");
constexpr size_t kStaticCbFloats = kStaticScratchFloats - kStaticFlagWords;
static_assert(kStaticCbFloats == SSM_STATIC_SCRATCH_FLOATS, "header and library disagree");

static __device__ __align__(256) float g_noalloc_scratch[kStaticScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float *g_noalloc_ptr[kMaxDevices] = {};
CUcontext g_noalloc_ctx[kMaxDevices] = {};
thread_local const char *g_noalloc_path = "none";

using CtxGetCurrent = CUresult (*)(CUcontext *);

// The driver's cuCtxGetCurrent, looked up through the runtime once per process.
CtxGetCurrent ctx_get_current() {
    static const CtxGetCurrent fn = []() -> CtxGetCurrent {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<CtxGetCurrent>(f);
    }();
    return fn;
}

// Device address of the scratch array on the current device.  In host code
// the array's name is only a stand-in for the symbol, so the address is
// looked up with the device current: once per device, and again whenever
// the device's context is not the one the address was taken in (after a
// cudaDeviceReset the runtime makes a new primary context, in which the
// library's module, and so the array, may sit at another address).
cudaError_t noalloc_scratch(float **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const CtxGetCurrent get = ctx_get_current();
    if (!get) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;  // null until the runtime has made the device's context current
    if (get(&ctx) != CUDA_SUCCESS) return cudaErrorNotSupported;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!ctx || !g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // also makes the primary context current
        if (e != cudaSuccess) return e;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorNotSupported;
        g_noalloc_ptr[dev] = static_cast<float *>(p);
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace ssm

extern "C" ssm_status ssm_verify_replay_static(int32_t batch, int32_t n_tok, int32_t nheads, int32_t headdim,
                                               int32_t dstate, int32_t ngroups, int32_t window, int32_t input_dtype,
                                               int32_t dt_dtype, const float *ckpt, void *log_x, float *log_dt,
                                               void *log_B, const int32_t *log_len, const void *x, const void *dt,
                                               const void *B, const void *C, const float *A, const float *D, void *y,
                                               uint32_t *flags, ssm_stream_t stream) {
    using namespace ssm;
    const bool n_ok = dstate == 16 || dstate == 32 || dstate == 64 || dstate == 128 || dstate == 256;
    if (batch < 1 || batch > kMaxSlotsPerLaunch || n_tok < 1 || n_tok > 64 || nheads < 1 || headdim < 1 ||
        headdim > 256 || !n_ok || ngroups < 1 || nheads % ngroups || window < 1 || window > 1024)
        return SSM_ERR_INVALID_ARG;
    if ((input_dtype != SSM_DTYPE_F32 && input_dtype != SSM_DTYPE_BF16) ||
        (dt_dtype != SSM_DTYPE_F32 && dt_dtype != SSM_DTYPE_BF16))
        return SSM_ERR_INVALID_ARG;
    if (!ckpt || !log_x || !log_dt || !log_B || !log_len || !x || !dt || !B || !C || !A || !D || !y || !flags)
        return SSM_ERR_INVALID_ARG;
    const int wcap = window - 1 + n_tok;
    const int cb_w = (wcap + 3) / 4 * 4;
    if ((size_t)batch * ngroups * n_tok * cb_w > kStaticCbFloats) return SSM_ERR_INVALID_ARG;  // scratch too small
    const int rows_per_warp = (32 / (dstate / 16)) * kRowsPerThread;
    if (32 * ((headdim + rows_per_warp - 1) / rows_per_warp) > kMaxThreads) return SSM_ERR_INVALID_ARG;

    // launch geometry only: a Pool describing the caller's buffers (no allocation)
    Pool view;
    view.device = 0;
    view.cfg.nheads = nheads; view.cfg.headdim = headdim; view.cfg.dstate = dstate; view.cfg.ngroups = ngroups;
    view.cfg.input_dtype = input_dtype; view.cfg.dt_dtype = dt_dtype; view.cfg.mode = SSM_MODE_REPLAY;
    view.cfg.window = window; view.cfg.max_tokens = n_tok;
    view.H = nheads; view.P = headdim; view.N = dstate; view.G = ngroups; view.hpg = nheads / ngroups;
    view.t1max = n_tok; view.wcap = wcap; view.n_slots = batch; view.cb_w = cb_w;
    int dev = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&view.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SSM_ERR_CUDA;
    view.device = dev;
    if (view.sm_count < 1) view.sm_count = 1;  // the persistent kernels size their grids by it
    if (replay_smem_bytes(view, n_tok) > (size_t)max_smem || replay_prep_smem_bytes(view, n_tok) > (size_t)max_smem)
        return SSM_ERR_INVALID_ARG;

    float *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return SSM_ERR_CUDA;
    uint32_t *req_flags = reinterpret_cast<uint32_t *>(scratch + kStaticCbFloats);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // per-request status words start clear on every call (the pair matrix
    // is fully rewritten for every pair the verify reads)
    if (cudaMemsetAsync(req_flags, 0, (size_t)batch * sizeof(uint32_t), s) != cudaSuccess) return SSM_ERR_CUDA;

    StepArgs a;
    std::memset(&a, 0, offsetof(StepArgs, slots));
    a.x = x; a.dt = dt; a.B = B; a.C = C; a.A = A; a.D = D; a.y = y;
    a.state = const_cast<float *>(ckpt);  // read only: the replay kernels never write the checkpoint
    a.log_x = log_x; a.log_dt = log_dt; a.log_B = log_B;
    a.cb = scratch;
    a.cb_w = cb_w;
    a.log_len = const_cast<int32_t *>(log_len);  // read only
    a.slot_flags = req_flags;
    a.flags = flags;
    a.H = nheads; a.P = headdim; a.N = dstate; a.G = ngroups; a.hpg = nheads / ngroups;
    a.n_slots = batch; a.t1max = n_tok; a.wcap = wcap;
    a.n_tok = n_tok;
    a.dt_bf16 = dt_dtype == SSM_DTYPE_BF16;
    a.check_log = 1;
    a.batch = batch;
    for (int i = 0; i < batch; ++i) a.slots[i] = i;  // request i owns row i of every caller buffer
    const char *path = "verify_replay";
    const cudaError_t e = launch_verify_replay(view, a, s, &path);
    g_noalloc_path = e == cudaSuccess ? path : "none";
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

namespace ssm {
const char *static_last_path() { return g_noalloc_path; }
}  // namespace ssm
