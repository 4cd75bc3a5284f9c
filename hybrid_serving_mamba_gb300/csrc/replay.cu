// ReplaySSM verify, and the commit of a verify step (copy and replay pools).
//
// Replay verify (Why Speculative Decoding Slows Hybrid Mamba Models, The
// Fix): with the checkpoint h_c, the k logged tokens and the step tokens
// u_k .. u_{k+n_tok-1} forming one token sequence u, the output of step
// token j (m = k + j + 1 tokens applied) is
//
//   y_j[p] = exp(A a_j) (C_j . h_c[p,:]) + sum_{s<m} W[j][s] x_s[p] + D x_j[p]
//   W[j][s] = exp(A a_{j,s}) dt_s (C_j . B_s)
//
// where a_j is the sum of all m applied dt and a_{j,s} the sum of the dt
// applied after token s.  The checkpoint is read once; each state element
// costs n_tok FMAs (the C_j . h_c products); the small W matrix and the
// log term W X are computed from shared memory.  No state is written.
//
// The commit (same page, The Fix, and The Problem for the copy flavour):
// copy pools move the slot's current-state index onto the snapshot of the
// last kept token; replay pools either append the kept tokens to the log or,
// when the window would fill, fold log + kept tokens into the checkpoint in
// closed form, h <- exp(A a) h + sum_s (exp(A a_s) dt_s x_s) (x) B_s.
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

struct ReplaySmem {
    float *B, *x, *C, *dt, *W, *decay, *d;
};

// Shared-memory carve-up for m token rows and n_tok step tokens.
// C and B first: N is a multiple of 16, so both stay 16-byte aligned for
// float4 reads whatever P is.
__host__ __device__ inline size_t replay_floats(int m, int n_tok, int N, int P) {
    return (size_t)n_tok * N + (size_t)m * N + (size_t)m * P + m + (size_t)n_tok * m + n_tok + (size_t)n_tok * P;
}

__device__ inline ReplaySmem carve(float *base, int m, int n_tok, int N, int P) {
    ReplaySmem s;
    s.C = base;
    s.B = s.C + (size_t)n_tok * N;
    s.x = s.B + (size_t)m * N;
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
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
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
    const TI *lB = reinterpret_cast<const TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    const float *ldt = a.log_dt + (size_t)slot * a.wcap * a.H;
    const TI *sx = reinterpret_cast<const TI *>(a.x);
    const TI *sB = reinterpret_cast<const TI *>(a.B);
    const TI *sC = reinterpret_cast<const TI *>(a.C);
    TI *wx = reinterpret_cast<TI *>(a.log_x) + (size_t)slot * a.wcap * a.H * P;
    TI *wB = reinterpret_cast<TI *>(a.log_B) + (size_t)slot * a.wcap * a.G * N;
    float *wdt = a.log_dt + (size_t)slot * a.wcap * a.H;

    // token sequence u = log[0..k) ++ step tokens, staged in shared memory;
    // the step tokens are also written after the log for the commit
    bool bad = false;
    for (int e = threadIdx.x; e < m * N; e += blockDim.x) {
        const int s = e / N, n = e - s * N;
        float b;
        if (s < k) {
            b = to_f(lB[((size_t)s * a.G + g) * N + n]);
        } else {
            const TI raw = sB[(((size_t)i * T1 + (s - k)) * a.G + g) * N + n];
            b = to_f(raw);
            bad |= !isfinite(b);
            if (h == g * a.hpg) wB[((size_t)s * a.G + g) * N + n] = raw;
        }
        sm.B[e] = b;
    }
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
    for (int e = threadIdx.x; e < T1 * N; e += blockDim.x) {
        const int j = e / N, n = e - j * N;
        const float c = to_f(sC[(((size_t)i * T1 + j) * a.G + g) * N + n]);
        bad |= !isfinite(c);
        sm.C[e] = c;
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
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }

    // decay weights: thread j accumulates the dt applied after each token,
    // from the newest token backwards (the time elapsed since token s)
    for (int j = threadIdx.x; j < T1; j += blockDim.x) {
        float after = 0.f;
        for (int s = k + j; s >= 0; --s) {
            sm.W[(size_t)j * m + s] = expf(A * after) * sm.dt[s];
            after += sm.dt[s];
        }
        for (int s = k + j + 1; s < m; ++s) sm.W[(size_t)j * m + s] = 0.f;
        sm.decay[j] = expf(A * after);
    }
    __syncthreads();
    // W[j][s] *= C_j . B_s for s <= k + j: one warp per pair, lanes over n
    for (int pr = warp; pr < T1 * m; pr += nwarps) {
        const int j = pr / m, s = pr - j * m;
        if (s > k + j) continue;
        float dot = 0.f;
        for (int n = lane; n < N; n += 32) dot = fmaf(sm.C[(size_t)j * N + n], sm.B[(size_t)s * N + n], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) sm.W[(size_t)j * m + s] *= dot;
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

    // y_j[p] = decay_j d_j[p] + sum_s W[j][s] x_s[p] + D x_j[p]
    TI *y = reinterpret_cast<TI *>(a.y);
    for (int e = threadIdx.x; e < T1 * P; e += blockDim.x) {
        const int j = e / P, p = e - j * P;
        float acc = sm.decay[j] * sm.d[e];
        const float *wj = sm.W + (size_t)j * m;
        for (int s = 0; s <= k + j; ++s) acc = fmaf(wj[s], sm.x[(size_t)s * P + p], acc);
        acc = fmaf(D, sm.x[(size_t)(k + j) * P + p], acc);
        y[(((size_t)i * T1 + j) * a.H + h) * P + p] = from_f<TI>(acc);
    }
}

// ------------------------------------------------------------------ commit

// Decision shared by the fold and metadata kernels: tokens committed (c)
// and whether the log is folded.  Returns false when the slot is skipped.
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

template <int N, typename TI>
__global__ void __launch_bounds__(kMaxThreads) fold_kernel(const __grid_constant__ CommitArgs a) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    extern __shared__ float4 smem4[];
    __shared__ int s_go, s_m;
    const int h = blockIdx.x, i = blockIdx.y;
    const int slot = a.slots[i];
    const int g = h / a.hpg;
    const int P = a.P;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, rw = lane / LPR;

    if (threadIdx.x == 0) {
        const int k = a.log_len[slot];
        int c = 0;
        bool fold = false;
        uint32_t err;
        const bool ok = commit_decision(a, i, slot, k, c, fold, err);
        s_go = ok && fold && k >= 0 && k + c <= a.wcap;
        s_m = k + c;
    }
    __syncthreads();
    if (!s_go) return;
    const int m = s_m;
    float *sB = reinterpret_cast<float *>(smem4);   // [m][N]
    float *sxw = sB + (size_t)m * N;                 // [m][P]  w_s x_s[p]
    float *sdt = sxw + (size_t)m * P;                // [m]
    float *sw = sdt + m;                             // [m]
    __shared__ float s_decay;

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
    if (threadIdx.x == 0) {  // time elapsed after each token, newest first
        float after = 0.f;
        for (int s = m - 1; s >= 0; --s) {
            sw[s] = expf(A * after) * sdt[s];
            after += sdt[s];
        }
        s_decay = expf(A * after);
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
}

// One thread per request: the index side of the commit (bit exact).
__global__ void commit_meta_kernel(const __grid_constant__ CommitArgs a, int replay) {
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
        a.log_len[slot] = fold ? 0 : k + c;
    } else {
        const int cur = a.cur[slot];
        const int half = (cur >= 0 && cur < a.t1max) ? 1 : 0;  // the half the verify wrote
        a.cur[slot] = half * a.t1max + (c - 1);
    }
    a.position[slot] += c;
}

}  // namespace

size_t replay_smem_bytes(const Pool &pool, int n_tok) {
    const int m = pool.wcap - pool.t1max + n_tok;  // W - 1 + n_tok
    return replay_floats(m, n_tok, pool.N, pool.P) * sizeof(float);
}

size_t fold_smem_bytes(const Pool &pool) {
    const int m = pool.wcap;
    return ((size_t)m * pool.N + (size_t)m * pool.P + 2 * (size_t)m) * sizeof(float);
}

template <typename K>
static cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_verify_replay(const Pool &pool, const StepArgs &a, cudaStream_t s) {
    const dim3 grid(a.H, a.batch);
    const size_t smem = replay_smem_bytes(pool, a.n_tok);
    const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
    SSM_DISPATCH_N(a.N, {
        const dim3 block(32 * warps_for<NN>(a.P));
        if (bf) {
            auto k = verify_replay_kernel<NN, __nv_bfloat16>;
            cudaError_t e = set_smem(k, smem);
            if (e != cudaSuccess) return e;
            k<<<grid, block, smem, s>>>(a);
        } else {
            auto k = verify_replay_kernel<NN, float>;
            cudaError_t e = set_smem(k, smem);
            if (e != cudaSuccess) return e;
            k<<<grid, block, smem, s>>>(a);
        }
    });
    return cudaGetLastError();
}

cudaError_t launch_commit(const Pool &pool, const CommitArgs &a, cudaStream_t s) {
    const bool replay = pool.cfg.mode == SSM_MODE_REPLAY;
    if (replay) {
        const dim3 grid(a.H, a.batch);
        const size_t smem = fold_smem_bytes(pool);
        const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
        SSM_DISPATCH_N(a.N, {
            const dim3 block(32 * warps_for<NN>(a.P));
            if (bf) {
                auto k = fold_kernel<NN, __nv_bfloat16>;
                cudaError_t e = set_smem(k, smem);
                if (e != cudaSuccess) return e;
                k<<<grid, block, smem, s>>>(a);
            } else {
                auto k = fold_kernel<NN, float>;
                cudaError_t e = set_smem(k, smem);
                if (e != cudaSuccess) return e;
                k<<<grid, block, smem, s>>>(a);
            }
        });
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    commit_meta_kernel<<<(a.batch + 127) / 128, 128, 0, s>>>(a, replay ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace ssm
