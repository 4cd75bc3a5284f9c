// Chunked scan on the tensor cores: the Mamba-2 matrix ("state space
// duality") form (Mamba Streaming State That Survives Chunking, Separate
// Mamba-2 algebra from kernel behavior: the dual view lets prefill use the
// parallel structure inside a chunk while the recurrent state crosses
// chunks).  One CTA of 128 threads walks one (sequence, head) chain in
// kernel chunks of Q = 128 tokens, with the head's fp32 state in registers
// (thread n holds column n of the 64 x 128 state).  Per chunk, with
// cum_i = A * (dt_0 + ... + dt_i) over the chunk:
//
//   CB      = C B^T                                    (128 x 128, K = 128)
//   M[i][j] = CB[i][j] exp(cum_i - cum_j) dt_j, j <= i  (CUDA cores, to bf16)
//   Y       = M X                                      (128 x 64,  K = 128)
//   Z       = C S^T           (S = state before the chunk, bf16 copy)
//   dS^T    = B^T (w o X)     w_j = exp(cum_last - cum_j) dt_j
//   y_i     = Y_i + exp(cum_i) Z_i + D x_i
//   S      <- exp(cum_last) S + dS
//
// All four products are tcgen05.mma kind::f16 (bf16 operands from shared
// memory in the 128-byte-swizzled K-major layout, fp32 accumulators in
// TMEM, M = 128).  x, B and C are bf16 inputs, so C B^T and the X operands
// are exact; M, w o X and the state copy are rounded to bf16, the state
// itself stays fp32.  Tokens past the end of a sequence are zero rows.
#include "ssm_internal.cuh"
#include "tc.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int Q = 128, SP = 64, SN = 128;
constexpr uint32_t kTile128 = 128 * 128;  // bytes of one K-tile (64 bf16) of a 128-row operand
constexpr uint32_t kTile64 = 64 * 128;    // ... of a 64-row operand
constexpr uint32_t OFF_C = 0;                         // C   [i][n]   rows i, K = n   (2 K-tiles)
constexpr uint32_t OFF_B = OFF_C + 2 * kTile128;      // B   [j][n]   rows j, K = n
constexpr uint32_t OFF_BT = OFF_B + 2 * kTile128;     // B^T [n][j]   rows n, K = j
constexpr uint32_t OFF_M = OFF_BT + 2 * kTile128;     // M   [i][j]   rows i, K = j
constexpr uint32_t OFF_XT = OFF_M + 2 * kTile128;     // X^T [p][j]   rows p, K = j
constexpr uint32_t OFF_XW = OFF_XT + 2 * kTile64;     // (w o X)^T [p][j]
constexpr uint32_t OFF_S = OFF_XW + 2 * kTile64;      // S   [p][n]   rows p, K = n
constexpr uint32_t OFF_MISC = OFF_S + 2 * kTile64;    // cum[128], dt[128], warp sums, mbarrier, tmem base
constexpr uint32_t kSsdSmem = OFF_MISC + 2048 + 1024; // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 256;  // [0,128) C B^T, then Z in [0,64) and dS^T in [64,128); Y in [128,192)

// Byte offset of element (r, k) of an operand whose K spans two 64-wide tiles.
__device__ __forceinline__ uint32_t opnd_off(uint32_t tile_bytes, uint32_t r, uint32_t k) {
    return (k >> 6) * tile_bytes + tc::sw128_offset(r, k & 63u);
}

__device__ __forceinline__ void st_bf16(unsigned char *base, uint32_t off, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(v);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
}

// K = 128 product of two swizzled operands into TMEM (8 MMAs of K = 16).
__device__ __forceinline__ void mma_k128(uint32_t d_tmem, uint32_t a_base, uint32_t a_tile, uint32_t b_base,
                                         uint32_t b_tile, uint32_t idesc) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (uint32_t)(ks & 3) * 32u;  // 16 bf16 along K inside the 128-byte row
        const uint64_t a = tc::smem_desc_sw128(a_base + (uint32_t)(ks >> 2) * a_tile + koff, 1024);
        const uint64_t b = tc::smem_desc_sw128(b_base + (uint32_t)(ks >> 2) * b_tile + koff, 1024);
        tc::mma_bf16(d_tmem, a, b, idesc, ks > 0);
    }
}

template <typename TI>
__global__ void __launch_bounds__(128, 1) scan_ssd_kernel(const __grid_constant__ ScanArgs a) {
    static_assert(sizeof(TI) == 2, "tensor-core scan takes bf16 x, B and C");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);
    float *s_cum = reinterpret_cast<float *>(smem + OFF_MISC);         // [128]
    float *s_dt = s_cum + Q;                                           // [128]
    float *s_wsum = s_dt + Q;                                          // [4]
    uint64_t *s_bar = reinterpret_cast<uint64_t *>(smem + OFF_MISC + 1056);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + OFF_MISC + 1072);
    uint32_t *s_gate = s_tmem + 1;

    const int h = blockIdx.x, i_seq = blockIdx.y;
    const int t0 = a.cu[i_seq], t1 = a.cu[i_seq + 1];
    if (t1 <= t0) return;  // empty chunk: consumes its sequence number only
    const int slot = a.slots[i_seq];
    const int H = a.H, G = a.G, g = h / a.hpg;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        uint32_t gate = 0;
        if (a.slot_flags[slot] & kSlotPoisoned) gate = SSM_FLAG_POISONED_SLOT;
        else if (a.check_log && a.log_len[slot] != 0) gate = SSM_FLAG_LOG_NOT_EMPTY;
        *s_gate = gate;
        mbar_init(s_bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    const uint32_t gate = *s_gate;
    if (gate) {
        if (tid == 0) {
            atomicOr(a.flags, gate);
            if (gate != SSM_FLAG_POISONED_SLOT) atomicOr(a.slot_flags + slot, kSlotPoisoned);
        }
        return;
    }
    if (warp == 0) tc::tmem_alloc(s_tmem, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;  // this warp's TMEM lane quadrant

    const float A = a.A[h], D = a.D[h];
    const TI *xg = reinterpret_cast<const TI *>(a.x);
    const TI *Bg = reinterpret_cast<const TI *>(a.B);
    const TI *Cg = reinterpret_cast<const TI *>(a.C);
    TI *yg = reinterpret_cast<TI *>(a.y);
    float *st = current_state(a.state, a.snap, a.cur, a.n_slots, (size_t)H * SP * SN, (size_t)SP * SN, slot, h);

    // state: thread n holds S[p][n] for all p, and writes the bf16 copy
    float S[SP];
#pragma unroll
    for (int p = 0; p < SP; ++p) S[p] = st[(size_t)p * SN + tid];
#pragma unroll
    for (int p = 0; p < SP; ++p) st_bf16(smem, OFF_S + opnd_off(kTile64, p, tid), S[p]);

    constexpr uint32_t kIdN128 = tc::idesc_bf16_f32(128, 128);
    constexpr uint32_t kIdN64 = tc::idesc_bf16_f32(128, 64);
    uint32_t phase = 0;
    bool bad = false, timeout = false;
    const int L = t1 - t0;
    for (int c0 = 0; c0 < L && !timeout; c0 += Q) {
        const int len = L - c0 < Q ? L - c0 : Q;
        const int t = tid;
        const bool valid = t < len;
        const size_t tok = (size_t)(t0 + c0 + t);

        // ---- P1: inputs of row t; dt prefix sums
        uint4 xr[8];
        float dtv = 0.f;
        if (valid) {
            const uint4 *xs = reinterpret_cast<const uint4 *>(xg + (tok * H + h) * SP);
#pragma unroll
            for (int c = 0; c < 8; ++c) xr[c] = xs[c];
            dtv = load_dt(a.dt, tok * H + h, a.dt_bf16);
            const uint4 *cs = reinterpret_cast<const uint4 *>(Cg + (tok * G + g) * SN);
            const uint4 *bs = reinterpret_cast<const uint4 *>(Bg + (tok * G + g) * SN);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 cv = cs[c], bv = bs[c];
                const uint32_t off = (uint32_t)(c >> 3) * kTile128 + (uint32_t)t * 128u +
                                     ((((uint32_t)c & 7u) ^ ((uint32_t)t & 7u)) << 4);
                *reinterpret_cast<uint4 *>(smem + OFF_C + off) = cv;
                *reinterpret_cast<uint4 *>(smem + OFF_B + off) = bv;
                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
                const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 bf = unpack_bf16(bw[e]), cf = unpack_bf16(cw[e]);
                    bad |= !isfinite(bf.x) || !isfinite(bf.y) || !isfinite(cf.x) || !isfinite(cf.y);
                    const uint32_t n = (uint32_t)c * 8u + 2u * e;
                    // B^T: row n, column (K) t
                    *reinterpret_cast<uint16_t *>(smem + OFF_BT + opnd_off(kTile128, n, t)) = (uint16_t)(bw[e] & 0xFFFFu);
                    *reinterpret_cast<uint16_t *>(smem + OFF_BT + opnd_off(kTile128, n + 1, t)) = (uint16_t)(bw[e] >> 16);
                }
            }
            bad |= !isfinite(dtv);
        } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) xr[c] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t off = (uint32_t)(c >> 3) * kTile128 + (uint32_t)t * 128u +
                                     ((((uint32_t)c & 7u) ^ ((uint32_t)t & 7u)) << 4);
                *reinterpret_cast<uint4 *>(smem + OFF_C + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(smem + OFF_B + off) = make_uint4(0, 0, 0, 0);
            }
#pragma unroll 8
            for (int n = 0; n < SN; ++n) *reinterpret_cast<uint16_t *>(smem + OFF_BT + opnd_off(kTile128, n, t)) = 0;
        }
        // inclusive prefix sum of dt over the chunk's 128 rows
        float v = dtv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) s_wsum[warp] = v;
        s_dt[t] = dtv;
        __syncthreads();
        for (int w = 0; w < warp; ++w) v += s_wsum[w];
        const float cum = A * v;
        s_cum[t] = cum;
        __syncthreads();
        const float cum_last = s_cum[Q - 1];
        const float wt = expf(cum_last - cum) * dtv;  // weight of token t in the state update
        // X^T and (w o X)^T: column t
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t xw[4] = {xr[c].x, xr[c].y, xr[c].z, xr[c].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xf = unpack_bf16(xw[e]);
                bad |= !isfinite(xf.x) || !isfinite(xf.y);
                const uint32_t p = (uint32_t)c * 8u + 2u * e;
                *reinterpret_cast<uint16_t *>(smem + OFF_XT + opnd_off(kTile64, p, t)) = (uint16_t)(xw[e] & 0xFFFFu);
                *reinterpret_cast<uint16_t *>(smem + OFF_XT + opnd_off(kTile64, p + 1, t)) = (uint16_t)(xw[e] >> 16);
                st_bf16(smem, OFF_XW + opnd_off(kTile64, p, t), xf.x * wt);
                st_bf16(smem, OFF_XW + opnd_off(kTile64, p + 1, t), xf.y * wt);
            }
        }
        tc::fence_proxy_async_smem();
        __syncthreads();

        // ---- P2: C B^T
        if (tid == 0) {
            tc::fence_after_sync();
            mma_k128(tmem, sbase + OFF_C, kTile128, sbase + OFF_B, kTile128, kIdN128);
            tc::mma_commit(s_bar);
        }
        if (__syncthreads_or(!mbar_wait(s_bar, phase & 1u))) {  // uniform across the CTA
            timeout = true;
            break;
        }
        ++phase;
        tc::fence_after_sync();

        // ---- P3: M = C B^T o decay o dt, masked to j <= i (row i = tid)
#pragma unroll 1
        for (int jb = 0; jb < Q; jb += 32) {
            float cb[32];
            tc::tmem_ld32(tmem + lane_addr + (uint32_t)jb, cb);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float mv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int j = jb + q8 * 8 + 2 * e + u;
                        mv[u] = j <= t ? cb[q8 * 8 + 2 * e + u] * expf(cum - s_cum[j]) * s_dt[j] : 0.f;
                    }
                    pk[e] = pack_bf16(mv[0], mv[1]);
                }
                const uint32_t j0 = (uint32_t)(jb + q8 * 8);
                *reinterpret_cast<uint4 *>(smem + OFF_M + opnd_off(kTile128, t, j0)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        tc::fence_before_sync();
        tc::fence_proxy_async_smem();
        __syncthreads();

        // ---- P4: Y = M X, Z = C S^T, dS^T = B^T (w o X)
        if (tid == 0) {
            tc::fence_after_sync();
            mma_k128(tmem + 128, sbase + OFF_M, kTile128, sbase + OFF_XT, kTile64, kIdN64);
            mma_k128(tmem + 0, sbase + OFF_C, kTile128, sbase + OFF_S, kTile64, kIdN64);
            mma_k128(tmem + 64, sbase + OFF_BT, kTile128, sbase + OFF_XW, kTile64, kIdN64);
            tc::mma_commit(s_bar);
        }
        if (__syncthreads_or(!mbar_wait(s_bar, phase & 1u))) {
            timeout = true;
            break;
        }
        ++phase;
        tc::fence_after_sync();

        // ---- P5: outputs of row t, and the state update of column n = t
        const float ecum = expf(cum);
        const float dA = expf(cum_last);
#pragma unroll
        for (int pb = 0; pb < SP; pb += 32) {
            float yv[32], zv[32], ds[32];
            tc::tmem_ld32(tmem + lane_addr + 128u + (uint32_t)pb, yv);
            tc::tmem_ld32(tmem + lane_addr + 0u + (uint32_t)pb, zv);
            tc::tmem_ld32(tmem + lane_addr + 64u + (uint32_t)pb, ds);
            uint32_t out[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int c = (pb + 2 * e) >> 3, w4 = ((pb + 2 * e) & 7) >> 1;
                const uint32_t xwv = w4 == 0 ? xr[c].x : w4 == 1 ? xr[c].y : w4 == 2 ? xr[c].z : xr[c].w;
                const float2 xf = unpack_bf16(xwv);
                const float y0 = fmaf(ecum, zv[2 * e], yv[2 * e]) + D * xf.x;
                const float y1 = fmaf(ecum, zv[2 * e + 1], yv[2 * e + 1]) + D * xf.y;
                out[e] = pack_bf16(y0, y1);
            }
            if (valid) {
                uint4 *yo = reinterpret_cast<uint4 *>(yg + (tok * H + h) * SP + pb);
#pragma unroll
                for (int c = 0; c < 4; ++c) yo[c] = make_uint4(out[4 * c], out[4 * c + 1], out[4 * c + 2], out[4 * c + 3]);
            }
#pragma unroll
            for (int p = 0; p < 32; ++p) S[pb + p] = fmaf(dA, S[pb + p], ds[p]);
        }
#pragma unroll
        for (int p = 0; p < SP; ++p) st_bf16(smem, OFF_S + opnd_off(kTile64, p, tid), S[p]);
        tc::fence_before_sync();
        tc::fence_proxy_async_smem();
        __syncthreads();
    }

    const bool any_bad = __syncthreads_or(bad);
    if (!any_bad && !timeout) {
#pragma unroll
        for (int p = 0; p < SP; ++p) st[(size_t)p * SN + tid] = S[p];
        if (h == 0 && tid == 0) a.position[slot] += L;
    } else if (tid == 0) {
        atomicOr(a.flags, timeout ? SSM_FLAG_TIMEOUT : SSM_FLAG_NONFINITE_INPUT);
        atomicOr(a.slot_flags + slot, kSlotPoisoned);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool scan_ssd_supported(const Pool &pool) {
    return pool.cfg.input_dtype == SSM_DTYPE_BF16 && pool.P == SP && pool.N == SN;
}

cudaError_t launch_scan_ssd(const Pool &pool, const ScanArgs &a, cudaStream_t s) {
    (void)pool;
    auto k = scan_ssd_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSsdSmem);
    if (e != cudaSuccess) return e;
    k<<<dim3(a.H, a.n_seq), 128, kSsdSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ssm
