// Decode step, copy verify, state gather and slot reset.
//
// Decode (batched single-token incremental update; Mamba Streaming State
// That Survives Chunking, Separate Mamba-2 algebra from kernel behavior) and
// copy verify (Why Speculative Decoding Slows Hybrid Mamba Models, The
// Problem) stream every state byte through registers exactly once in and
// once (decode) or n_tok times (copy verify) out; they are HBM-bound with
// 2-3 FMAs per 4-byte element.  See ssm_internal.cuh for the lane layout.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int RPT = kRowsPerThread;

template <int N>
__host__ __device__ constexpr int rows_per_warp() { return 32 / (N / 16); }

template <int N>
int warps_for(int P) {
    const int rows = rows_per_warp<N>() * RPT;
    return (P + rows - 1) / rows;
}

// Slot-level gate shared by every state kernel: returns the SSM_FLAG_* bit
// that forbids work on this slot (0 = go).  Read by thread 0 only.
__device__ __forceinline__ uint32_t slot_gate(const uint32_t *slot_flags, const int32_t *log_len,
                                              int check_log, int slot) {
    if (slot_flags[slot] & kSlotPoisoned) return SSM_FLAG_POISONED_SLOT;
    if (check_log && log_len[slot] != 0) return SSM_FLAG_LOG_NOT_EMPTY;
    return 0;
}

__device__ __forceinline__ void raise_flag(uint32_t *flags, uint32_t *slot_flags, int slot, uint32_t bit) {
    atomicOr(flags, bit);
    if (bit != SSM_FLAG_POISONED_SLOT) atomicOr(slot_flags + slot, kSlotPoisoned);
}

// ------------------------------------------------------------------ decode

// MAXT / MINB: launch bounds.  CTAs of up to 256 threads are compiled for
// three per SM (at most 85 registers a thread): more state loads in flight.
template <int N, typename TI, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) decode_kernel(const __grid_constant__ StepArgs a) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    __shared__ uint32_t s_gate;
    const int h = blockIdx.x, i = blockIdx.y;
    const int slot = a.slots[i];
    const int g = h / a.hpg;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, rw = lane / LPR;
    if (threadIdx.x == 0) s_gate = slot_gate(a.slot_flags, a.log_len, a.check_log, slot);

    float *st = current_state(a.state, a.snap, a.cur, a.n_slots, (size_t)a.H * a.P * N, (size_t)a.P * N, slot, h);
    const TI *x = reinterpret_cast<const TI *>(a.x) + ((size_t)i * a.H + h) * a.P;

    // state rows first: the loads that matter are in flight while the rest arrives
    float4 v[RPT][4];
    float xv[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int p = (warp * RPT + k) * RPW + rw;
        if (p < a.P) {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[k][q] = ld_stream(st + (size_t)p * N + 4 * (sub + LPR * q));
            xv[k] = to_f(x[p]);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[k][q] = make_float4(0.f, 0.f, 0.f, 0.f);
            xv[k] = 0.f;
        }
    }
    float Bv[16], Cv[16];
    load_lane16<N>(reinterpret_cast<const TI *>(a.B) + ((size_t)i * a.G + g) * N, sub, Bv);
    load_lane16<N>(reinterpret_cast<const TI *>(a.C) + ((size_t)i * a.G + g) * N, sub, Cv);
    const float dt = load_dt(a.dt, (size_t)i * a.H + h, a.dt_bf16);
    const float A = a.A[h], D = a.D[h];

    bool bad = !isfinite(dt);
#pragma unroll
    for (int e = 0; e < 16; ++e) bad |= !isfinite(Bv[e]) || !isfinite(Cv[e]);
#pragma unroll
    for (int k = 0; k < RPT; ++k) bad |= !isfinite(xv[k]);
    __syncthreads();
    const uint32_t gate = s_gate;
    if (gate) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, gate);
        return;
    }
    if (__syncthreads_or(bad)) {  // nothing advances: the state is not written
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
        return;
    }

    const float dA = expf(dt * A);
    TI *y = reinterpret_cast<TI *>(a.y) + ((size_t)i * a.H + h) * a.P;
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int p = (warp * RPT + k) * RPW + rw;
        const float dtx = dt * xv[k];
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float4 &w = v[k][q];
            w.x = fmaf(dA, w.x, dtx * Bv[4 * q + 0]); acc = fmaf(Cv[4 * q + 0], w.x, acc);
            w.y = fmaf(dA, w.y, dtx * Bv[4 * q + 1]); acc = fmaf(Cv[4 * q + 1], w.y, acc);
            w.z = fmaf(dA, w.z, dtx * Bv[4 * q + 2]); acc = fmaf(Cv[4 * q + 2], w.z, acc);
            w.w = fmaf(dA, w.w, dtx * Bv[4 * q + 3]); acc = fmaf(Cv[4 * q + 3], w.w, acc);
        }
        acc = row_sum<LPR>(acc);
        if (p < a.P) {
#pragma unroll
            for (int q = 0; q < 4; ++q) st_stream(st + (size_t)p * N + 4 * (sub + LPR * q), v[k][q]);
            if (sub == 0) y[p] = from_f<TI>(fmaf(D, xv[k], acc));
        }
    }
    if (h == 0 && threadIdx.x == 0) a.position[slot] += 1;
}

// ------------------------------------------------------------------ copy verify

template <int N, typename TI, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) verify_copy_kernel(const __grid_constant__ StepArgs a) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    __shared__ uint32_t s_gate;
    const int h = blockIdx.x, i = blockIdx.y;
    const int slot = a.slots[i];
    const int g = h / a.hpg;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, rw = lane / LPR;
    if (threadIdx.x == 0) s_gate = slot_gate(a.slot_flags, a.log_len, 0, slot);

    const int cur = a.cur[slot];
    const int half = (cur >= 0 && cur < a.t1max) ? 1 : 0;  // never overwrite the current state
    const float *src = current_state(a.state, a.snap, a.cur, a.n_slots, (size_t)a.H * a.P * N, (size_t)a.P * N, slot, h);
    const size_t slot_stride = (size_t)a.n_slots * a.H * a.P * N;
    float *dst0 = a.snap + (size_t)half * a.t1max * slot_stride + ((size_t)slot * a.H + h) * (size_t)a.P * N;

    float4 v[RPT][4];
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
        const int p = (warp * RPT + k) * RPW + rw;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            v[k][q] = p < a.P ? ld_stream(src + (size_t)p * N + 4 * (sub + LPR * q)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float A = a.A[h], D = a.D[h];
    __syncthreads();
    const uint32_t gate = s_gate;
    if (gate) {
        if (threadIdx.x == 0) raise_flag(a.flags, a.slot_flags, slot, gate);
        return;
    }

    bool bad = false;
    for (int j = 0; j < a.n_tok; ++j) {
        const size_t tok = (size_t)i * a.n_tok + j;
        float Bv[16], Cv[16];
        load_lane16<N>(reinterpret_cast<const TI *>(a.B) + (tok * a.G + g) * N, sub, Bv);
        load_lane16<N>(reinterpret_cast<const TI *>(a.C) + (tok * a.G + g) * N, sub, Cv);
        const float dt = load_dt(a.dt, tok * a.H + h, a.dt_bf16);
        const TI *x = reinterpret_cast<const TI *>(a.x) + (tok * a.H + h) * a.P;
        TI *y = reinterpret_cast<TI *>(a.y) + (tok * a.H + h) * a.P;
        float *dst = dst0 + (size_t)j * slot_stride;
        const float dA = expf(dt * A);
        bad |= !isfinite(dt);
#pragma unroll
        for (int e = 0; e < 16; ++e) bad |= !isfinite(Bv[e]) || !isfinite(Cv[e]);
#pragma unroll
        for (int k = 0; k < RPT; ++k) {
            const int p = (warp * RPT + k) * RPW + rw;
            const float xv = p < a.P ? to_f(x[p]) : 0.f;
            bad |= !isfinite(xv);
            const float dtx = dt * xv;
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 &w = v[k][q];
                w.x = fmaf(dA, w.x, dtx * Bv[4 * q + 0]); acc = fmaf(Cv[4 * q + 0], w.x, acc);
                w.y = fmaf(dA, w.y, dtx * Bv[4 * q + 1]); acc = fmaf(Cv[4 * q + 1], w.y, acc);
                w.z = fmaf(dA, w.z, dtx * Bv[4 * q + 2]); acc = fmaf(Cv[4 * q + 2], w.z, acc);
                w.w = fmaf(dA, w.w, dtx * Bv[4 * q + 3]); acc = fmaf(Cv[4 * q + 3], w.w, acc);
            }
            acc = row_sum<LPR>(acc);
            if (p < a.P) {
#pragma unroll
                for (int q = 0; q < 4; ++q) st_stream(dst + (size_t)p * N + 4 * (sub + LPR * q), v[k][q]);
                if (sub == 0) y[p] = from_f<TI>(fmaf(D, xv, acc));
            }
        }
    }
    // snapshots are scratch until commit; a bad input poisons the slot so
    // that the commit of this step is refused
    if (__syncthreads_or(bad) && threadIdx.x == 0)
        raise_flag(a.flags, a.slot_flags, slot, SSM_FLAG_NONFINITE_INPUT);
}

// ------------------------------------------------------------------ gather / reset

struct SlotList {
    int32_t slots[kMaxSlotsPerLaunch];
};

__global__ void gather_kernel(const float *state, const float *snap, const int32_t *cur, int n_slots,
                              size_t hpn, int has_snap, const __grid_constant__ SlotList l, float *dst) {
    const int i = blockIdx.y;
    const int slot = l.slots[i];
    const float *src = state + (size_t)slot * hpn;
    if (has_snap) {
        const int c = cur[slot];
        if (c >= 0) src = snap + ((size_t)c * n_slots + slot) * hpn;
    }
    float *d = dst + (size_t)i * hpn;
    const size_t n4 = hpn / 4;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4; e += (size_t)gridDim.x * blockDim.x)
        reinterpret_cast<float4 *>(d)[e] = reinterpret_cast<const float4 *>(src)[e];
}

__global__ void reset_kernel(float *state, size_t hpn, int64_t *position, int32_t *log_len, int32_t *cur,
                             uint32_t *slot_flags, const __grid_constant__ SlotList l) {
    const int i = blockIdx.y;
    const int slot = l.slots[i];
    float4 *d = reinterpret_cast<float4 *>(state + (size_t)slot * hpn);
    const size_t n4 = hpn / 4;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4; e += (size_t)gridDim.x * blockDim.x)
        d[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        position[slot] = 0;
        log_len[slot] = 0;
        if (cur) cur[slot] = -1;
        slot_flags[slot] = 0;
    }
}

}  // namespace

// ------------------------------------------------------------------ launchers

// Launch K<N, TI, 256, 3> for CTAs of at most 256 threads, else K<N, TI, kMaxThreads, 1>.
#define SSM_LAUNCH_BOUNDED(K, NN, TI, grid, block, s, a)                       \
    do {                                                                        \
        if ((block).x <= 256) K<NN, TI, 256, 3><<<grid, block, 0, s>>>(a);      \
        else K<NN, TI, kMaxThreads, 1><<<grid, block, 0, s>>>(a);               \
    } while (0)

cudaError_t launch_decode(const Pool &pool, const StepArgs &a, cudaStream_t s) {
    const dim3 grid(a.H, a.batch);
    const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
    SSM_DISPATCH_N(a.N, {
        const dim3 block(32 * warps_for<NN>(a.P));
        if (bf) SSM_LAUNCH_BOUNDED(decode_kernel, NN, __nv_bfloat16, grid, block, s, a);
        else SSM_LAUNCH_BOUNDED(decode_kernel, NN, float, grid, block, s, a);
    });
    return cudaGetLastError();
}

cudaError_t launch_verify_copy(const Pool &pool, const StepArgs &a, cudaStream_t s) {
    const dim3 grid(a.H, a.batch);
    const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
    SSM_DISPATCH_N(a.N, {
        const dim3 block(32 * warps_for<NN>(a.P));
        if (bf) SSM_LAUNCH_BOUNDED(verify_copy_kernel, NN, __nv_bfloat16, grid, block, s, a);
        else SSM_LAUNCH_BOUNDED(verify_copy_kernel, NN, float, grid, block, s, a);
    });
    return cudaGetLastError();
}

cudaError_t launch_gather(const Pool &pool, const int32_t *slots, int n, float *dst, cudaStream_t s) {
    for (int base = 0; base < n; base += kMaxSlotsPerLaunch) {
        const int m = n - base < kMaxSlotsPerLaunch ? n - base : kMaxSlotsPerLaunch;
        SlotList l;
        for (int i = 0; i < m; ++i) l.slots[i] = slots[base + i];
        const int bx = (int)((pool.hpn / 4 + 255) / 256 < 64 ? (pool.hpn / 4 + 255) / 256 : 64);
        gather_kernel<<<dim3(bx, m), 256, 0, s>>>(pool.state, pool.snap, pool.d_cur, pool.n_slots, pool.hpn,
                                                  pool.snap != nullptr, l, dst + (size_t)base * pool.hpn);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_reset(const Pool &pool, const int32_t *slots, int n, cudaStream_t s) {
    for (int base = 0; base < n; base += kMaxSlotsPerLaunch) {
        const int m = n - base < kMaxSlotsPerLaunch ? n - base : kMaxSlotsPerLaunch;
        SlotList l;
        for (int i = 0; i < m; ++i) l.slots[i] = slots[base + i];
        const int bx = (int)((pool.hpn / 4 + 255) / 256 < 64 ? (pool.hpn / 4 + 255) / 256 : 64);
        reset_kernel<<<dim3(bx, m), 256, 0, s>>>(pool.state, pool.hpn, pool.d_position, pool.d_log_len,
                                                 pool.d_cur, pool.d_slot_flags, l);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ssm
