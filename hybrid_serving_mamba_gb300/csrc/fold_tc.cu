// ReplaySSM fold on the tensor cores (Why Speculative Decoding Slows Hybrid
// Mamba Models, The Fix: once the window fills, the checkpoint takes the
// logged tokens and the log empties).  For a folding request with m logged
// tokens and one head:
//
//   h <- d h + sum_{s < m} (w_s x_s) (x) B_s,
//   d = exp(A sum_{s < m} dt_s),  w_s = exp(A sum_{s < r < m} dt_r) dt_s,
//
// a rank-m update of the P x N fp32 checkpoint.  An item is a pair of heads
// (h0, h0 + 1) of one request (the same group, so the same logged B rows):
// D = W B on the tensor cores with W[row][s] = w_s x_s[p] for the 128 rows
// (head, p) and B[s][n] the group's logged rows, K = KP (the longest window
// rounded up to 32, 48 or 64; zero past m), then h <- d h + D row by row.
//
// W is fp32; it enters kind::f16 MMAs as three bf16 terms hi = rn(v),
// mid = rn(v - hi), lo = rn(v - hi - mid), whose sum carries 24 significant
// bits as fp32 does, and B is bf16 as logged, so the fold keeps the state at
// fp32 accuracy with 3 KP / 16 MMAs (M = 128, N = 128, K = 16) per item.
//
// Warps: 0-3 rows (thread = row 32 w + lane, TMEM lane quarter w): the head's
//          dt prefix sums and w_s, W into TMEM, then h <- d h + D in place in
//          the staged checkpoint tile;
//        4 producer (lane 0): the checkpoint (four 32-column TMA boxes of the
//          two heads' 128 rows), the logged x rows of both heads and KP
//          logged B rows of the group (two 64-column boxes, 128-byte swizzle:
//          the MMA's MN-major B tile) into a two-stage ring; it also stores
//          each finished checkpoint back by TMA before reusing its stage;
//        5 MMA issuer (lane 0) and TMEM owner.
// TMEM: D of stage s at columns 128 s; W of stage s at 256 + (3 KP / 2) s
// (hi in columns 0 .. KP/2 - 1, mid in the next KP/2, lo in the last KP/2,
// two bf16 of consecutive s per column, the lower s in the low half).
#include "ssm_internal.cuh"
#include "tc.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kFtRowWarps = 4;
constexpr int kFtProd = 4, kFtMma = 5;
constexpr int kFtThreads = 6 * 32;
constexpr int kFtStages = 2;
constexpr uint32_t kFtBox = 16384;           // 32 fp32 columns x 128 rows
constexpr uint32_t kFtHBytes = 4 * kFtBox;   // both heads' checkpoints
constexpr uint32_t kFtCols = 512;
static_assert(256 + kFtStages * 3 * kMaxFoldK / 2 <= (int)kFtCols, "D and W of both stages fit in TMEM");

struct FtLayout {
    uint32_t bbox, b, x, stage, bars, total;
};

// Per stage: checkpoint boxes, B boxes of kp rows x 128 bytes (1024-aligned
// for the swizzle), the two heads' logged x rows [wwin][2][P] bf16; after the
// stages the barriers.
__host__ __device__ inline FtLayout ft_layout(int wcap, int P, int kp) {
    FtLayout L;
    L.bbox = (uint32_t)kp * 128u;
    L.b = kFtHBytes;
    L.x = L.b + 2u * L.bbox;
    const uint32_t end = L.x + (uint32_t)wcap * 2u * (uint32_t)P * 2u;
    L.stage = (end + 1023u) & ~1023u;
    L.bars = kFtStages * L.stage;
    L.total = L.bars + 4 * kFtStages * 8 + 1024;  // full, wful, done, hful; + alignment of the base
    return L;
}

__device__ __forceinline__ bool ft_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort, uint32_t *flags) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && *abort) return false;
    }
    *abort = 1u;
    atomicOr(flags, SSM_FLAG_TIMEOUT);
    return false;
}

// The row warps' barrier (named barrier 1, 128 threads) that ORs a predicate.
__device__ __forceinline__ bool rows_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(kFtRowWarps * 32)
        : "memory");
    return r != 0;
}

// The (slot, first head, group, m) of item `item`.
struct FtItem {
    int slot, h0, g, m;
};
__device__ __forceinline__ FtItem ft_item(const CommitArgs &a, int item) {
    const int hp = a.H / 2;
    const int f = item / hp;
    const int2 it = a.fold_items[f];
    FtItem r;
    r.h0 = 2 * (item - f * hp);
    r.slot = a.slots[it.x];
    r.g = r.h0 / a.hpg;
    r.m = it.y;
    return r;
}

// Store n (a multiple of 8) consecutive 32-bit TMEM columns of this thread's lane.
template <int n>
__device__ __forceinline__ void ft_store_cols(uint32_t taddr, const uint32_t *v) {
#pragma unroll
    for (int c = 0; c + 16 <= n; c += 16) tc::tmem_st16(taddr + c, *reinterpret_cast<const uint32_t(*)[16]>(v + c));
    if constexpr (n % 16 != 0) tc::tmem_st8(taddr + (n - 8), v + (n - 8));
}

// KP: the K extent (32, 48 or 64), at least the longest window.
template <int KP>
__global__ void __launch_bounds__(kFtThreads, 1)
    fold_tc_kernel(const __grid_constant__ CommitArgs a, const __grid_constant__ CUtensorMap tm_state,
                   const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b) {
    static_assert(KP % 16 == 0 && KP >= 32 && KP <= kMaxFoldK, "");
    constexpr int KC = KP / 2;  // TMEM columns of one W term
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t s_abort, s_tmem;
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    // the next verify's coefficient kernel may be scheduled as this grid drains (it waits for it)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int P = a.P, H = a.H;
    const FtLayout L = ft_layout(a.wwin, P, KP);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);  // tiles landed
    uint64_t *wful = full + kFtStages;                              // W in TMEM, B tile trimmed
    uint64_t *done = wful + kFtStages;                              // MMAs finished
    uint64_t *hful = done + kFtStages;                              // new checkpoint in the tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = *a.fold_count * (H / 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kFtStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&wful[s], kFtRowWarps);
            mbar_init(&done[s], 1);
            mbar_init(&hful[s], kFtRowWarps);
        }
        mbar_fence_init();
        s_abort = 0u;
    }
    if (warp == kFtMma) tc::tmem_alloc(&s_tmem, kFtCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    if (warp == kFtProd) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t bytes = kFtHBytes + 2u * L.bbox + (uint32_t)a.wwin * 2u * (uint32_t)P * 2u;
            int loaded[kFtStages];
            for (int s = 0; s < kFtStages; ++s) loaded[s] = -1;
            bool alive = true;
            // item v's new checkpoint back to the pool, once its rows have written it
            auto store = [&](int v) -> bool {
                const int st = v % kFtStages;
                if (!ft_wait(&hful[st], (uint32_t)(v / kFtStages) & 1u, &s_abort, a.flags)) return false;
                const FtItem it = ft_item(a, blockIdx.x + v * gridDim.x);
                const unsigned char *S = smem + (size_t)st * L.stage;
                const int row0 = (it.slot * H + it.h0) * P;
                for (int kb = 0; kb < 4; ++kb) tma_store_2d(&tm_state, kb * 32, row0, S + kb * kFtBox);
                bulk_commit();
                bulk_wait_read0();  // the tile may be refilled
                return true;
            };
            int u = 0;
            for (;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int st = u % kFtStages;
                if (u >= kFtStages && !store(u - kFtStages)) {
                    alive = false;
                    break;
                }
                const FtItem it = ft_item(a, item);
                unsigned char *S = smem + (size_t)st * L.stage;
                mbar_arrive_expect_tx(&full[st], bytes);
                const int row0 = (it.slot * H + it.h0) * P;
                for (int kb = 0; kb < 4; ++kb) tma_load_2d(S + kb * kFtBox, &tm_state, kb * 32, row0, &full[st]);
                tma_load_3d(S + L.b, &tm_b, 0, it.g, it.slot * a.wcap, &full[st]);
                tma_load_3d(S + L.b + L.bbox, &tm_b, 64, it.g, it.slot * a.wcap, &full[st]);
                tma_load_3d(S + L.x, &tm_x, 0, it.h0, it.slot * a.wcap, &full[st]);
                loaded[st] = u;
            }
            for (int v = u > kFtStages ? u - kFtStages : 0; alive && v < u; ++v) alive = store(v);
            bulk_wait0();  // every store has completed
            // no load may still be landing when the CTA exits
            for (int s = 0; s < kFtStages; ++s)
                if (loaded[s] >= 0 && !mbar_wait(&full[s], (uint32_t)(loaded[s] / kFtStages) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp == kFtMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 128) | (1u << 16);  // B MN-major
            int last = -1;
            for (int u = 0;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int st = u % kFtStages;
                if (!ft_wait(&wful[st], (uint32_t)(u / kFtStages) & 1u, &s_abort, a.flags)) break;
                tc::fence_after_sync();
                const uint32_t d = tmem + 128u * st, w = tmem + 256u + (uint32_t)(3 * KC) * st;
                const uint32_t bbase = smem_addr(smem + (size_t)st * L.stage + L.b);
#pragma unroll
                for (int ks = 0; ks < KP / 16; ++ks) {  // K = 16: rows 16 ks .. of the B tile, 8 columns of W
                    const uint64_t bd = tc::smem_desc_sw128_lbo(bbase + 2048u * ks, L.bbox, 1024);
                    tc::mma_bf16_ta(d, w + 8 * ks, bd, idesc, ks > 0);
                    tc::mma_bf16_ta(d, w + KC + 8 * ks, bd, idesc, true);
                    tc::mma_bf16_ta(d, w + 2 * KC + 8 * ks, bd, idesc, true);
                }
                tc::mma_commit(&done[st]);
                last = u;
            }
            // every MMA issued has completed before TMEM is released
            if (last >= 0 && !mbar_wait(&done[last % kFtStages], (uint32_t)(last / kFtStages) & 1u))
                atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ rows
        const int row = threadIdx.x, hd = row >> 6, p = row & 63;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        for (int u = 0;; ++u) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            const int st = u % kFtStages;
            const FtItem it = ft_item(a, item);
            const int h = it.h0 + hd, m = it.m;  // 1 <= m <= wwin <= KP
            const float A = a.A[h];
            // dt of the head's logged tokens s = lane (and s = lane + 32 when KP > 32); prefix sums as
            // fp32 pairs, so that each difference is as exact as fp32 can hold
            const float *ldt = a.log_dt + (size_t)it.slot * a.wcap * H + h;
            const float dt0 = lane < m ? ldt[(size_t)lane * H] : 0.f;
            const float dt1 = (KP > 32 && lane + 32 < m) ? ldt[(size_t)(lane + 32) * H] : 0.f;
            Sum2 c0{dt0, 0.f}, c1{dt1, 0.f};
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const Sum2 q0{__shfl_up_sync(0xffffffffu, c0.hi, o), __shfl_up_sync(0xffffffffu, c0.lo, o)};
                if (lane >= o) c0 = sum2_add(q0, c0);
                if constexpr (KP > 32) {
                    const Sum2 q1{__shfl_up_sync(0xffffffffu, c1.hi, o), __shfl_up_sync(0xffffffffu, c1.lo, o)};
                    if (lane >= o) c1 = sum2_add(q1, c1);
                }
            }
            if constexpr (KP > 32)
                c1 = sum2_add(Sum2{__shfl_sync(0xffffffffu, c0.hi, 31), __shfl_sync(0xffffffffu, c0.lo, 31)}, c1);
            const int last = m - 1;
            const Sum2 t0{__shfl_sync(0xffffffffu, c0.hi, last & 31), __shfl_sync(0xffffffffu, c0.lo, last & 31)};
            const Sum2 t1{__shfl_sync(0xffffffffu, c1.hi, last & 31), __shfl_sync(0xffffffffu, c1.lo, last & 31)};
            const Sum2 tot = last < 32 ? t0 : t1;
            const float ws0 = lane < m ? expf(A * sum2_diff(tot, c0)) * dt0 : 0.f;  // w_s at s = lane
            const float ws1 = lane + 32 < m ? expf(A * sum2_diff(tot, c1)) * dt1 : 0.f;
            const float decay = expf(A * (tot.hi + tot.lo));

            const bool ok = ft_wait(&full[st], (uint32_t)(u / kFtStages) & 1u, &s_abort, a.flags);
            if (rows_or(!ok)) break;
            unsigned char *S = smem + (size_t)st * L.stage;
            // B rows s >= m hold other log entries: zero them (whole 128-byte rows of both boxes)
            for (int e = row; e < (KP - m) * 16; e += kFtRowWarps * 32) {
                const int r = m + (e >> 4), c = e & 15;
                *reinterpret_cast<uint4 *>(S + L.b + (uint32_t)(c >> 3) * L.bbox + (uint32_t)r * 128u +
                                           ((uint32_t)(c & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            }
            // W[row][s] = w_s x_s[p] for s < m (zero beyond), as bf16 hi / mid / lo of pairs of s
            const __nv_bfloat16 *xr = reinterpret_cast<const __nv_bfloat16 *>(S + L.x) + hd * P + p;
            uint32_t hi[KC], mid[KC], lo[KC];
#pragma unroll
            for (int c = 0; c < KC; ++c) {
                float v[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int s = 2 * c + e;
                    const float wsv = __shfl_sync(0xffffffffu, s < 32 ? ws0 : ws1, s & 31);
                    v[e] = s < m ? wsv * __bfloat162float(xr[(size_t)s * 2 * P]) : 0.f;
                }
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[0], v[1]);
                const float r0 = v[0] - __low2float(h2), r1 = v[1] - __high2float(h2);
                const __nv_bfloat162 m2 = __floats2bfloat162_rn(r0, r1);
                const __nv_bfloat162 l2 = __floats2bfloat162_rn(r0 - __low2float(m2), r1 - __high2float(m2));
                hi[c] = *reinterpret_cast<const uint32_t *>(&h2);
                mid[c] = *reinterpret_cast<const uint32_t *>(&m2);
                lo[c] = *reinterpret_cast<const uint32_t *>(&l2);
            }
            const uint32_t w = tmem + lane_off + 256u + (uint32_t)(3 * KC) * st;
            ft_store_cols<KC>(w, hi);
            ft_store_cols<KC>(w + KC, mid);
            ft_store_cols<KC>(w + 2 * KC, lo);
            tc::tmem_wait_st();
            tc::fence_proxy_async_smem();  // the zeroed B rows, for the MMA
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&wful[st]);

            // h <- d h + D, in place in the staged checkpoint tile
            const bool okd = ft_wait(&done[st], (uint32_t)(u / kFtStages) & 1u, &s_abort, a.flags);
            if (rows_or(!okd)) break;
            tc::fence_after_sync();
#pragma unroll 1
            for (int kb = 0; kb < 4; ++kb) {
                float dv[32];
                tc::tmem_ld32(tmem + lane_off + 128u * st + 32u * kb, dv);
                unsigned char *blk = S + (uint32_t)kb * kFtBox + (uint32_t)row * 128u;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {  // chunk ch of the row at ch ^ (row % 8)
                    float4 *q = reinterpret_cast<float4 *>(blk + ((uint32_t)(ch ^ (row & 7)) << 4));
                    float4 hv = *q;
                    hv.x = fmaf(decay, hv.x, dv[4 * ch + 0]);
                    hv.y = fmaf(decay, hv.y, dv[4 * ch + 1]);
                    hv.z = fmaf(decay, hv.z, dv[4 * ch + 2]);
                    hv.w = fmaf(decay, hv.w, dv[4 * ch + 3]);
                    *q = hv;
                }
            }
            tc::fence_before_sync();       // D read, before the MMA of the stage's next item
            tc::fence_proxy_async_smem();  // the new tile, for the TMA store
            __syncwarp();
            if (lane == 0) mbar_arrive(&hful[st]);
        }
    }
    __syncwarp();  // warps whose lane 0 ran a role alone arrive at the block barrier converged
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kFtMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kFtCols);
    }
}

}  // namespace

cudaError_t launch_fold_tc(const Pool &pool, const CommitArgs &a, cudaStream_t s) {
    const int kp = pool.fold_kp;
    if (!pool.tm_fold_ok || a.P != 64 || a.N != 128 || a.wwin > kp || (a.H & 1) || (a.hpg & 1))
        return cudaErrorNotSupported;
    const FtLayout L = ft_layout(a.wwin, a.P, kp);
    int dev = 0, max_smem = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (L.total > (uint32_t)max_smem) return cudaErrorNotSupported;
    auto launch = [&](auto kernel) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (e != cudaSuccess) return e;
        kernel<<<pool.sm_count, kFtThreads, L.total, s>>>(a, pool.tm_state2, pool.tm_logx2, pool.tm_logB);
        return cudaGetLastError();
    };
    switch (kp) {
    case 32: return launch(fold_tc_kernel<32>);
    case 48: return launch(fold_tc_kernel<48>);
    case 64: return launch(fold_tc_kernel<64>);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace ssm
