// Chunked scan, sequential form: one CTA per (sequence, head) walks the
// sequence's tokens in order with the head's state held in registers, and
// writes the final state back to the slot (Mamba Streaming State That
// Survives Chunking, Let the full scan define legal chunking: a chunk starts
// from the state its predecessor left).  Used for fp32 inputs (whose
// tolerance the bf16 tensor-core path cannot meet) and for shapes the
// tensor-core path does not cover.
//
// A chunk with a non-finite input leaves its slot's state untouched (the
// state is only stored after the whole chunk was seen) and poisons the slot.
#include "ssm_internal.cuh"

namespace ssm {
namespace {

constexpr int RPT = kRowsPerThread;

template <int N>
int warps_for(int P) {
    const int rows = (32 / (N / 16)) * RPT;
    return (P + rows - 1) / rows;
}

template <int N, typename TI>
struct TokenIn {
    float B[16], C[16], x[RPT], dt;
};

template <int N, typename TI>
__device__ __forceinline__ void load_token(const ScanArgs &a, size_t t, int h, int g, int sub, const int (&prow)[RPT],
                                           TokenIn<N, TI> &in) {
    load_lane16<N>(reinterpret_cast<const TI *>(a.B) + (t * a.G + g) * N, sub, in.B);
    load_lane16<N>(reinterpret_cast<const TI *>(a.C) + (t * a.G + g) * N, sub, in.C);
    in.dt = load_dt(a.dt, t * a.H + h, a.dt_bf16);
    const TI *x = reinterpret_cast<const TI *>(a.x) + (t * a.H + h) * a.P;
#pragma unroll
    for (int r = 0; r < RPT; ++r) in.x[r] = prow[r] >= 0 ? to_f(x[prow[r]]) : 0.f;
}

template <int N, typename TI>
__global__ void __launch_bounds__(kMaxThreads) scan_seq_kernel(const __grid_constant__ ScanArgs a) {
    constexpr int LPR = N / 16, RPW = 32 / LPR;
    __shared__ uint32_t s_gate;
    const int h = blockIdx.x, i = blockIdx.y;
    const int t0 = a.cu[i], t1 = a.cu[i + 1];
    if (t1 <= t0) return;  // empty chunk: consumes its sequence number only
    const int slot = a.slots[i];
    const int g = h / a.hpg;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, rw = lane / LPR;
    if (threadIdx.x == 0) {
        uint32_t gate = 0;
        if (a.slot_flags[slot] & kSlotPoisoned) gate = SSM_FLAG_POISONED_SLOT;
        else if (a.check_log && a.log_len[slot] != 0) gate = SSM_FLAG_LOG_NOT_EMPTY;
        s_gate = gate;
    }
    int prow[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int p = (warp * RPT + r) * RPW + rw;
        prow[r] = p < a.P ? p : -1;
    }
    float *st = current_state(a.state, a.snap, a.cur, a.n_slots, (size_t)a.H * a.P * N, (size_t)a.P * N, slot, h);
    float4 v[RPT][4];
#pragma unroll
    for (int r = 0; r < RPT; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q)
            v[r][q] = prow[r] >= 0 ? *reinterpret_cast<const float4 *>(st + (size_t)prow[r] * N + 4 * (sub + LPR * q))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    const float A = a.A[h], D = a.D[h];
    __syncthreads();
    const uint32_t gate = s_gate;
    if (gate) {
        if (threadIdx.x == 0) {
            atomicOr(a.flags, gate);
            if (gate != SSM_FLAG_POISONED_SLOT) atomicOr(a.slot_flags + slot, kSlotPoisoned);
        }
        return;
    }

    TI *y = reinterpret_cast<TI *>(a.y);
    bool bad = false;
    TokenIn<N, TI> cur, nxt;
    load_token<N, TI>(a, (size_t)t0, h, g, sub, prow, cur);
    for (int t = t0; t < t1; ++t) {
        if (t + 1 < t1) load_token<N, TI>(a, (size_t)t + 1, h, g, sub, prow, nxt);  // prefetch
        const float dA = expf(cur.dt * A);
        bad |= !isfinite(cur.dt);
#pragma unroll
        for (int e = 0; e < 16; ++e) bad |= !isfinite(cur.B[e]) || !isfinite(cur.C[e]);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            bad |= !isfinite(cur.x[r]);
            const float dtx = cur.dt * cur.x[r];
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 &w = v[r][q];
                w.x = fmaf(dA, w.x, dtx * cur.B[4 * q + 0]); acc = fmaf(cur.C[4 * q + 0], w.x, acc);
                w.y = fmaf(dA, w.y, dtx * cur.B[4 * q + 1]); acc = fmaf(cur.C[4 * q + 1], w.y, acc);
                w.z = fmaf(dA, w.z, dtx * cur.B[4 * q + 2]); acc = fmaf(cur.C[4 * q + 2], w.z, acc);
                w.w = fmaf(dA, w.w, dtx * cur.B[4 * q + 3]); acc = fmaf(cur.C[4 * q + 3], w.w, acc);
            }
            acc = row_sum<LPR>(acc);
            if (sub == 0 && prow[r] >= 0)
                y[((size_t)t * a.H + h) * a.P + prow[r]] = from_f<TI>(fmaf(D, cur.x[r], acc));
        }
        cur = nxt;
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) {
            atomicOr(a.flags, SSM_FLAG_NONFINITE_INPUT);
            atomicOr(a.slot_flags + slot, kSlotPoisoned);
        }
        return;
    }
#pragma unroll
    for (int r = 0; r < RPT; ++r)
        if (prow[r] >= 0)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<float4 *>(st + (size_t)prow[r] * N + 4 * (sub + LPR * q)) = v[r][q];
    if (h == 0 && threadIdx.x == 0) a.position[slot] += t1 - t0;
}

}  // namespace

cudaError_t launch_scan_seq(const Pool &pool, const ScanArgs &a, cudaStream_t s) {
    const dim3 grid(a.H, a.n_seq);
    const bool bf = pool.cfg.input_dtype == SSM_DTYPE_BF16;
    SSM_DISPATCH_N(a.N, {
        const dim3 block(32 * warps_for<NN>(a.P));
        if (bf) scan_seq_kernel<NN, __nv_bfloat16><<<grid, block, 0, s>>>(a);
        else scan_seq_kernel<NN, float><<<grid, block, 0, s>>>(a);
    });
    return cudaGetLastError();
}

}  // namespace ssm
