// ReplaySSM verify that folds a full log on the way (Why Speculative
// Decoding Slows Hybrid Mamba Models, The Fix: the checkpoint takes the
// logged tokens once the window is full; every verify reads the checkpoint
// anyway).  For a request whose log holds k >= W tokens, one head, and the
// n_tok step tokens j:
//
//   h'  = d h + sum_{s < k} (w_s x_s) (x) B_s           the fold (k logged tokens)
//   y_j = dec'_j (C_j . h') + sum_{s <= j} W'[j][s] x_{k+s}[p]
//
// with d, w_s the decay and weights of the logged tokens (as the fold at a
// commit), dec'_j and W' (D on its diagonal) the step's own coefficients,
// formed by the coefficient kernel as for a request with an empty log, and
// the step's rows staged after the log (rows k ..).  h' goes back as the
// checkpoint, so the request pays one checkpoint read and one write where a
// fold at the commit and the next verify would pay two reads and a write.
//
// An item is a pair of heads (h0, h0 + 1) of one listed request: their 128
// checkpoint rows (head, p) form the M of both products.
//   fold:    F = Xw B on the tensor cores, Xw[row][s] = w_s x_s[p] as bf16
//            hi / mid / lo (24 significant bits) in TMEM, B the logged rows
//            (bf16, MN-major tile), K = KP; then h' = d h + F row by row;
//   outputs: h' as bf16 hi + lo (16 significant bits) in the TMEM columns F
//            held, times C (bf16, K-major tile) into NM columns;
//   epilogue: y_j = dec'_j D[j] + the step's own term.
//
// Warps: 0-3 and 4-7 two row groups (thread = row 32 (w % 4) + lane, TMEM
//          lane quarter w % 4), group g taking the items of stage g, so that
//          one group's serial chain (weights, Xw, h', epilogue) overlaps the
//          other's;
//        8 producer (lane 0): per item the checkpoint (four 32-column boxes),
//          KP logged B rows of the group (two 64-column boxes), both heads'
//          whole logs of x rows, C in the operand layout, W' and dec' rows,
//          into a two-stage ring; it stores each new checkpoint back by TMA as
//          soon as its rows have written it, and reloads a stage once the
//          store has read the tile and the rows are done with the stage;
//        9, 10 MMA issuers (lane 0) of stages 0 and 1; 9 owns TMEM.
// TMEM per stage s: F, then the hi / lo of h', at columns 128 s; Xw at
// 256 + 3 KC s (hi, mid, lo of KC columns each), then D of the outputs there.
// A request whose slot is poisoned is computed but nothing of it is written
// (checkpoint, outputs, log length); the flag is raised.
#include "ssm_internal.cuh"
#include "tc.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int kFvRowWarps = 4;                         // per row group
constexpr int kFvStages = 2;                           // one per row group
constexpr int kFvProd = kFvStages * kFvRowWarps;       // 8
constexpr int kFvMma = kFvProd + 1;                    // 9 (stage 0, TMEM owner) and 10 (stage 1)
constexpr int kFvThreads = (kFvMma + kFvStages) * 32;  // 352
constexpr uint32_t kFvBox = 16384;           // 32 fp32 columns x 128 rows
constexpr uint32_t kFvHBytes = 4 * kFvBox;   // both heads' checkpoints
constexpr uint32_t kFvCols = 512;
static_assert(256 + kFvStages * 3 * kMaxFoldK / 2 <= (int)kFvCols, "F and Xw of both stages fit in TMEM");

__device__ __forceinline__ void raise_flag(uint32_t *flags, uint32_t *slot_flags, int slot, uint32_t bit) {
    atomicOr(flags, bit);
    if (bit != SSM_FLAG_POISONED_SLOT) atomicOr(slot_flags + slot, kSlotPoisoned);
}

struct FvLayout {
    uint32_t bbox, b, x, c, w, dec, stage, bars, total;
};

// Per stage (1024-aligned parts for the swizzled tiles): checkpoint boxes,
// B boxes of kp rows x 128 bytes, C as NM rows of each 64-column block, the
// two heads' logged x rows [wcap][2][P] bf16, W' [2][t1max][cb_w] and dec'
// [2][t1pad] fp32; after the stages the barriers.
__host__ __device__ inline FvLayout fv_layout(int wcap, int P, int kp, int NM, int t1max, int cb_w, int t1pad) {
    FvLayout L;
    L.bbox = (uint32_t)kp * 128u;
    L.b = kFvHBytes;
    L.c = L.b + 2u * L.bbox;                      // a multiple of 1024
    L.x = L.c + 2u * (uint32_t)NM * 128u;
    L.w = L.x + (((uint32_t)wcap * 2u * (uint32_t)P * 2u + 15u) & ~15u);
    L.dec = L.w + 2u * (uint32_t)t1max * (uint32_t)cb_w * 4u;
    const uint32_t end = L.dec + 2u * (uint32_t)t1pad * 4u;
    L.stage = (end + 1023u) & ~1023u;
    L.bars = kFvStages * L.stage;
    L.total = L.bars + 6 * kFvStages * 8 + 1024;  // full, wful, done, aful, ydone, hful; + alignment of the base
    return L;
}

__device__ __forceinline__ bool fv_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort, uint32_t *flags) {
    for (uint32_t it = 0; it < kWaitLimit; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 255u && *abort) return false;
    }
    *abort = 1u;
    atomicOr(flags, SSM_FLAG_TIMEOUT);
    return false;
}

// One row group's barrier (named barrier 1 + group, 128 threads) that ORs a predicate.
__device__ __forceinline__ bool fv_rows_or(int group, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(1 + group), "r"(kFvRowWarps * 32)
        : "memory");
    return r != 0;
}

struct FvItem {
    int i, slot, h0, g, k;
    bool poisoned;
};
__device__ __forceinline__ FvItem fv_item(const StepArgs &a, int item) {
    const int hp = a.H / 2;
    const int f = item / hp;
    const int2 it = a.fv_items[f];
    FvItem r;
    r.i = it.x;
    r.k = it.y;
    r.h0 = 2 * (item - f * hp);
    r.slot = a.slots[it.x];
    r.g = r.h0 / a.hpg;
    r.poisoned = (a.slot_flags[r.slot] & kSlotPoisoned) != 0;
    return r;
}

template <int n>
__device__ __forceinline__ void fv_store_cols(uint32_t taddr, const uint32_t *v) {
#pragma unroll
    for (int c = 0; c + 16 <= n; c += 16) tc::tmem_st16(taddr + c, *reinterpret_cast<const uint32_t(*)[16]>(v + c));
    if constexpr (n % 16 != 0) tc::tmem_st8(taddr + (n - 8), v + (n - 8));
}

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) { return *reinterpret_cast<const uint32_t *>(&v); }

// KP: K extent of the fold (32, 48 or 64, at least the longest log); NM: columns of the outputs (16 or 32).
template <int KP, int NM>
__global__ void __launch_bounds__(kFvThreads, 1)
    fold_verify_tc_kernel(const __grid_constant__ StepArgs a, const __grid_constant__ CUtensorMap tm_state,
                          const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b) {
    static_assert(KP % 16 == 0 && KP >= 32 && KP <= kMaxFoldK && (NM == 16 || NM == 32), "");
    constexpr int KC = KP / 2;  // TMEM columns of one Xw term
    static_assert(NM <= 3 * KC, "the outputs' D fits where Xw was");
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t s_abort, s_tmem;
    unsigned char *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int P = a.P, H = a.H, N = a.N, T1 = a.n_tok;
    const FvLayout L = fv_layout(a.wcap, P, KP, NM, a.t1max, a.cb_w, a.t1pad);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);  // tiles landed
    uint64_t *wful = full + kFvStages;                              // Xw in TMEM, B tile trimmed
    uint64_t *done = wful + kFvStages;                              // fold MMAs finished
    uint64_t *aful = done + kFvStages;                              // h' in the tile, its hi / lo in TMEM
    uint64_t *ydone = aful + kFvStages;                             // output MMAs finished
    uint64_t *hful = ydone + kFvStages;                             // the rows are done with the stage
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = *(volatile const int32_t *)&a.counts[1] * (H / 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kFvStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&wful[s], kFvRowWarps);
            mbar_init(&done[s], 1);
            mbar_init(&aful[s], kFvRowWarps);
            mbar_init(&ydone[s], 1);
            mbar_init(&hful[s], kFvRowWarps);
        }
        mbar_fence_init();
        s_abort = 0u;
    }
    if (warp == kFvMma) tc::tmem_alloc(&s_tmem, kFvCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;

    if (warp == kFvProd) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t cbytes = 2u * (uint32_t)NM * 128u;  // C: two 64-column blocks of NM rows
            const uint32_t bytes = kFvHBytes + 2u * L.bbox + cbytes + (uint32_t)a.wcap * 2u * (uint32_t)P * 2u +
                                   2u * a.t1max * a.cb_w * 4u + 2u * a.t1pad * 4u;
            int loaded[kFvStages];
            for (int s = 0; s < kFvStages; ++s) loaded[s] = -1;
            bool alive = true;
            // item v's new checkpoint back to the pool as soon as its rows have written it
            auto store = [&](int v) -> bool {
                const int st = v % kFvStages;
                if (!fv_wait(&aful[st], (uint32_t)(v / kFvStages) & 1u, &s_abort, a.flags)) return false;
                const FvItem it = fv_item(a, blockIdx.x + v * gridDim.x);
                if (!it.poisoned) {
                    const unsigned char *S = smem + (size_t)st * L.stage;
                    const int row0 = (it.slot * H + it.h0) * P;
                    for (int kb = 0; kb < 4; ++kb) tma_store_2d(&tm_state, kb * 32, row0, S + kb * kFvBox);
                    bulk_commit();
                }
                return true;
            };
            // item v's stage may be refilled: its rows are done and the store has read the tile
            auto reclaim = [&](int v) -> bool {
                if (!fv_wait(&hful[v % kFvStages], (uint32_t)(v / kFvStages) & 1u, &s_abort, a.flags)) return false;
                bulk_wait_read0();
                return true;
            };
            int u = 0;
            for (;; ++u) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int st = u % kFvStages;
                if (u >= kFvStages && !(store(u - kFvStages) && reclaim(u - kFvStages))) {
                    alive = false;
                    break;
                }
                const FvItem it = fv_item(a, item);
                unsigned char *S = smem + (size_t)st * L.stage;
                mbar_arrive_expect_tx(&full[st], bytes);
                const int row0 = (it.slot * H + it.h0) * P;
                for (int kb = 0; kb < 4; ++kb) tma_load_2d(S + kb * kFvBox, &tm_state, kb * 32, row0, &full[st]);
                tma_load_3d(S + L.b, &tm_b, 0, it.g, it.slot * a.wcap, &full[st]);
                tma_load_3d(S + L.b + L.bbox, &tm_b, 64, it.g, it.slot * a.wcap, &full[st]);
                tma_load_3d(S + L.x, &tm_x, 0, it.h0, it.slot * a.wcap, &full[st]);
                bulk_g2s(S + L.c, a.cf + ((size_t)it.i * a.G + it.g) * a.cf_rows * N, cbytes, &full[st]);
                bulk_g2s(S + L.w, a.wsc + ((size_t)it.i * H + it.h0) * a.t1max * a.cb_w, 2u * a.t1max * a.cb_w * 4u,
                         &full[st]);
                bulk_g2s(S + L.dec, a.dec + ((size_t)it.i * H + it.h0) * a.t1pad, 2u * a.t1pad * 4u, &full[st]);
                loaded[st] = u;
            }
            for (int v = u > kFvStages ? u - kFvStages : 0; alive && v < u; ++v) alive = store(v) && reclaim(v);
            bulk_wait0();  // every store has completed
            // no load may still be landing when the CTA exits
            for (int s = 0; s < kFvStages; ++s)
                if (loaded[s] >= 0 && !mbar_wait(&full[s], (uint32_t)(loaded[s] / kFvStages) & 1u))
                    atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else if (warp >= kFvMma) {
        // ------------------------------------------------------------ MMA issuers, one per stage
        if (lane == 0) {
            constexpr uint32_t idesc_f = tc::idesc_bf16_f32(128, 128) | (1u << 16);  // B MN-major
            constexpr uint32_t idesc_y = tc::idesc_bf16_f32(128, NM);
            int last = -1;
            for (int u = warp - kFvMma;; u += kFvStages) {
                const int item = blockIdx.x + u * gridDim.x;
                if (item >= n_items) break;
                const int st = u % kFvStages;
                const uint32_t ph = (uint32_t)(u / kFvStages) & 1u;
                const uint32_t f = tmem + 128u * st, w = tmem + 256u + (uint32_t)(3 * KC) * st;
                const unsigned char *S = smem + (size_t)st * L.stage;
                if (!fv_wait(&wful[st], ph, &s_abort, a.flags)) break;
                tc::fence_after_sync();
                const uint32_t bbase = smem_addr(S + L.b);
#pragma unroll
                for (int ks = 0; ks < KP / 16; ++ks) {  // K = 16: rows 16 ks .. of the B tile, 8 columns of Xw
                    const uint64_t bd = tc::smem_desc_sw128_lbo(bbase + 2048u * ks, L.bbox, 1024);
                    tc::mma_bf16_ta(f, w + 8 * ks, bd, idesc_f, ks > 0);
                    tc::mma_bf16_ta(f, w + KC + 8 * ks, bd, idesc_f, true);
                    tc::mma_bf16_ta(f, w + 2 * KC + 8 * ks, bd, idesc_f, true);
                }
                tc::mma_commit(&done[st]);
                last = u;
                // the outputs, once the rows have put h' where F was (they have read F and Xw by then)
                if (!fv_wait(&aful[st], ph, &s_abort, a.flags)) {
                    last = -1;  // F of this item was waited for by the rows, or they gave up
                    mbar_wait(&done[st], ph);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t cbase = smem_addr(S + L.c);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {  // K = 16 bf16 per MMA: 8 columns of hi (+0) and lo (+16)
                        const uint32_t boff = (uint32_t)(kb >> 1) * NM * 128 + (kb & 1) * 64 + 32 * kk;
                        const uint64_t bd = tc::smem_desc_sw128(cbase + boff, 1024);
                        const uint32_t at = f + 32u * kb;
                        tc::mma_bf16_ta(w, at + 8 * kk, bd, idesc_y, (kb | kk) != 0);
                        tc::mma_bf16_ta(w, at + 16 + 8 * kk, bd, idesc_y, true);
                    }
                }
                tc::mma_commit(&ydone[st]);
            }
            // every MMA issued has completed before TMEM is released
            if (last >= 0 && !mbar_wait(&ydone[last % kFvStages], (uint32_t)(last / kFvStages) & 1u))
                atomicOr(a.flags, SSM_FLAG_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ rows
        const int rg = warp / kFvRowWarps, q = warp % kFvRowWarps;  // row group (= its stage), lane quarter
        const int row = 32 * q + lane, hd = row >> 6, p = row & 63;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        __nv_bfloat16 *y = reinterpret_cast<__nv_bfloat16 *>(a.y);
        for (int u = rg;; u += kFvStages) {
            const int item = blockIdx.x + u * gridDim.x;
            if (item >= n_items) break;
            const int st = u % kFvStages;
            const uint32_t ph = (uint32_t)(u / kFvStages) & 1u;
            const FvItem it = fv_item(a, item);
            const int h = it.h0 + hd, k = it.k;  // W <= k <= the longest log <= KP
            const float A = a.A[h];
            // dt of the head's logged tokens s = lane (and s = lane + 32 when KP > 32); prefix sums as
            // fp32 pairs, so that each difference is as exact as fp32 can hold
            const float *ldt = a.log_dt + (size_t)it.slot * a.wcap * H + h;
            const float dt0 = lane < k ? ldt[(size_t)lane * H] : 0.f;
            const float dt1 = (KP > 32 && lane + 32 < k) ? ldt[(size_t)(lane + 32) * H] : 0.f;
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
            const int last = k - 1;
            const Sum2 t0{__shfl_sync(0xffffffffu, c0.hi, last & 31), __shfl_sync(0xffffffffu, c0.lo, last & 31)};
            const Sum2 t1{__shfl_sync(0xffffffffu, c1.hi, last & 31), __shfl_sync(0xffffffffu, c1.lo, last & 31)};
            const Sum2 tot = last < 32 ? t0 : t1;
            const float ws0 = lane < k ? expf(A * sum2_diff(tot, c0)) * dt0 : 0.f;  // w_s at s = lane
            const float ws1 = lane + 32 < k ? expf(A * sum2_diff(tot, c1)) * dt1 : 0.f;
            const float decay = expf(A * (tot.hi + tot.lo));

            const bool ok = fv_wait(&full[st], ph, &s_abort, a.flags);
            if (fv_rows_or(rg, !ok)) break;
            unsigned char *S = smem + (size_t)st * L.stage;
            // B rows s >= k hold the staged step and other log entries: zero them (whole 128-byte rows)
            for (int e = row; e < (KP - k) * 16; e += kFvRowWarps * 32) {
                const int r = k + (e >> 4), c = e & 15;
                *reinterpret_cast<uint4 *>(S + L.b + (uint32_t)(c >> 3) * L.bbox + (uint32_t)r * 128u +
                                           ((uint32_t)(c & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            }
            // Xw[row][s] = w_s x_s[p] for s < k (zero beyond), as bf16 hi / mid / lo of pairs of s
            const __nv_bfloat16 *xr = reinterpret_cast<const __nv_bfloat16 *>(S + L.x) + hd * P + p;
            {
                uint32_t hi[KC], mid[KC], lo[KC];
#pragma unroll
                for (int c = 0; c < KC; ++c) {
                    float v[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = 2 * c + e;
                        const float wsv = __shfl_sync(0xffffffffu, s < 32 ? ws0 : ws1, s & 31);
                        v[e] = s < k ? wsv * __bfloat162float(xr[(size_t)s * 2 * P]) : 0.f;
                    }
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[0], v[1]);
                    const float r0 = v[0] - __low2float(h2), r1 = v[1] - __high2float(h2);
                    const __nv_bfloat162 m2 = __floats2bfloat162_rn(r0, r1);
                    const __nv_bfloat162 l2 = __floats2bfloat162_rn(r0 - __low2float(m2), r1 - __high2float(m2));
                    hi[c] = bf2_bits(h2);
                    mid[c] = bf2_bits(m2);
                    lo[c] = bf2_bits(l2);
                }
                const uint32_t w = tmem + lane_off + 256u + (uint32_t)(3 * KC) * st;
                fv_store_cols<KC>(w, hi);
                fv_store_cols<KC>(w + KC, mid);
                fv_store_cols<KC>(w + 2 * KC, lo);
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async_smem();  // the zeroed B rows, for the MMA
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&wful[st]);

            // h' = d h + F in place in the staged tile, and h' as bf16 hi / lo where F was
            const bool okd = fv_wait(&done[st], ph, &s_abort, a.flags);
            if (fv_rows_or(rg, !okd)) break;
            tc::fence_after_sync();
            const uint32_t ft = tmem + lane_off + 128u * st;
#pragma unroll 1
            for (int kb = 0; kb < 4; ++kb) {
                float dv[32];
                tc::tmem_ld32(ft + 32u * kb, dv);
                unsigned char *blk = S + (uint32_t)kb * kFvBox + (uint32_t)row * 128u;
                uint32_t hl[32];  // columns 0-15: hi of elements (2c, 2c + 1); 16-31: lo of the same
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {  // chunk ch of the row at ch ^ (row % 8)
                    float4 *q = reinterpret_cast<float4 *>(blk + ((uint32_t)(ch ^ (row & 7)) << 4));
                    float4 hv = *q;
                    hv.x = fmaf(decay, hv.x, dv[4 * ch + 0]);
                    hv.y = fmaf(decay, hv.y, dv[4 * ch + 1]);
                    hv.z = fmaf(decay, hv.z, dv[4 * ch + 2]);
                    hv.w = fmaf(decay, hv.w, dv[4 * ch + 3]);
                    *q = hv;
                    const __nv_bfloat162 h0 = __floats2bfloat162_rn(hv.x, hv.y), h1 = __floats2bfloat162_rn(hv.z, hv.w);
                    const __nv_bfloat162 l0 = __floats2bfloat162_rn(hv.x - __low2float(h0), hv.y - __high2float(h0));
                    const __nv_bfloat162 l1 = __floats2bfloat162_rn(hv.z - __low2float(h1), hv.w - __high2float(h1));
                    hl[2 * ch] = bf2_bits(h0);
                    hl[2 * ch + 1] = bf2_bits(h1);
                    hl[16 + 2 * ch] = bf2_bits(l0);
                    hl[16 + 2 * ch + 1] = bf2_bits(l1);
                }
                tc::tmem_st32(ft + 32u * kb, hl);  // F of this block was read above (the load waits)
            }
            tc::fence_before_sync();
            tc::fence_proxy_async_smem();  // the new tile, for the TMA store
            __syncwarp();
            if (lane == 0) mbar_arrive(&aful[st]);

            // the step's own term while the output MMAs run: sum_{s <= j} W'[j][s] x_{k+s}[p]
            const float *Wh = reinterpret_cast<const float *>(S + L.w) + (size_t)hd * a.t1max * a.cb_w;
            const float *dh = reinterpret_cast<const float *>(S + L.dec) + (size_t)hd * a.t1pad;
            float lt[NM];
#pragma unroll
            for (int j = 0; j < NM; ++j) lt[j] = 0.f;
#pragma unroll 1
            for (int s = 0; s < T1; ++s) {
                const float xs = __bfloat162float(xr[(size_t)(k + s) * 2 * P]);
#pragma unroll
                for (int j = 0; j < NM; ++j)
                    if (j < T1 && s <= j) lt[j] = fmaf(Wh[(size_t)j * a.cb_w + s], xs, lt[j]);
            }
            const bool oky = fv_wait(&ydone[st], ph, &s_abort, a.flags);
            if (fv_rows_or(rg, !oky)) break;
            tc::fence_after_sync();
            float d[NM];
            const uint32_t dt_ = tmem + lane_off + 256u + (uint32_t)(3 * KC) * st;
#pragma unroll
            for (int c = 0; c < NM; c += 16) {
                float part[16];
                tc::tmem_ld16(dt_ + c, part);
#pragma unroll
                for (int q = 0; q < 16; ++q) d[c + q] = part[q];
            }
            if (it.poisoned) {
                if (row == 0) raise_flag(a.flags, a.slot_flags, it.slot, SSM_FLAG_POISONED_SLOT);
            } else {
                __nv_bfloat16 *yrow = y + ((size_t)it.i * T1 * H + h) * P + p;
#pragma unroll
                for (int j = 0; j < NM; ++j)
                    if (j < T1) yrow[(size_t)j * H * P] = __float2bfloat16_rn(fmaf(dh[j], d[j], lt[j]));
                if (it.h0 == 0 && row == 0) a.log_len[it.slot] = 0;  // the log is in the checkpoint now
            }
            tc::fence_before_sync();  // D read, before the stage's next item
            __syncwarp();
            if (lane == 0) mbar_arrive(&hful[st]);
        }
    }
    __syncwarp();  // warps whose lane 0 ran a role alone arrive at the block barrier converged
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kFvMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kFvCols);
    }
}

int fv_nm(int t1max) { return t1max <= 16 ? 16 : 32; }

}  // namespace

bool fold_verify_fits(const Pool &pool) {
    if (!pool.tm_fold_ok || pool.P != 64 || pool.N != 128 || pool.t1max > 32) return false;
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, pool.device);
    const FvLayout L = fv_layout(pool.wcap, pool.P, pool.fold_kp, fv_nm(pool.t1max), pool.t1max, pool.cb_w, pool.t1pad);
    return L.total <= (uint32_t)max_smem;
}

cudaError_t launch_fold_verify_tc(const Pool &pool, const StepArgs &a, int NM, cudaStream_t s) {
    const int kp = pool.fold_kp;
    if (!pool.tm_fold_ok || !pool.fold_in_verify || !a.fv_items || a.P != 64 || a.N != 128 || a.wwin > kp ||
        (a.H & 1) || (a.hpg & 1) || NM != fv_nm(pool.t1max) || a.cf_nm != NM)
        return cudaErrorNotSupported;
    const FvLayout L = fv_layout(a.wcap, a.P, kp, NM, a.t1max, a.cb_w, a.t1pad);
    auto launch = [&](auto kernel) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (e != cudaSuccess) return e;
        kernel<<<pool.sm_count, kFvThreads, L.total, s>>>(a, pool.tm_state2, pool.tm_logx_fv, pool.tm_logB);
        return cudaGetLastError();
    };
#define SSM_FV(KPV)                                                                       \
    case KPV:                                                                             \
        return NM == 16 ? launch(fold_verify_tc_kernel<KPV, 16>) : launch(fold_verify_tc_kernel<KPV, 32>)
    switch (kp) {
        SSM_FV(32);
        SSM_FV(48);
        SSM_FV(64);
    default: return cudaErrorNotSupported;
    }
#undef SSM_FV
}

}  // namespace ssm
