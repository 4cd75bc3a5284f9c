// Chunked scan on the tensor cores: the Mamba-2 matrix ("state space
// duality") form (Mamba Streaming State That Survives Chunking, Separate
// Mamba-2 algebra from kernel behavior: the dual view lets prefill use the
// parallel structure inside a chunk while the recurrent state crosses
// chunks).  One CTA of 256 threads walks one (sequence, head) chain in
// kernel chunks of Q = 128 tokens; the head's fp32 state stays in registers
// (thread (n, half) holds S[p][n] for the 32 rows p of its half).  Per chunk,
// with cum_i = A * (dt_0 + ... + dt_i) over the chunk:
//
//   CB      = C B^T                                    (128 x 128, K = 128)
//   M[i][j] = CB[i][j] exp(cum_i - cum_j) dt_j, j <= i  (CUDA cores, to bf16)
//   Y       = M X                                      (128 x 64,  K = 128)
//   Z       = C S^T           (S = state before the chunk, bf16 copy)
//   dS^T    = B^T (w o X)     w_j = exp(cum_last - cum_j) dt_j
//   y_i     = Y_i + exp(cum_i) Z_i + D x_i
//   S      <- exp(cum_last) S + dS
//
// All four products are tcgen05.mma kind::f16 with bf16 operands in
// 128-byte-swizzled shared-memory tiles and fp32 accumulators in TMEM
// (M = 128).  Operands are stored the way their producers write them -- one
// row per token (C, B, X, w o X) or per state column (S) -- and read K-major
// or MN-major as each product needs, so no transposes are made.  C B^T and Z
// go first, together: C and the state copy are then free, so M takes the
// place of C and w o X that of the state copy, which keeps a CTA at 100 KiB
// of shared memory, 256 TMEM columns and 128 registers a thread: two CTAs
// (two chains) share an SM and each one's waits on the tensor core and on
// memory overlap the other's work.  x, B and C
// are bf16 inputs, so C B^T and X are exact; M, w o X and the state copy
// are rounded to bf16, the state itself stays fp32.
//
// Non-finite inputs are found where they surface, in y and in the state
// increment (each input enters one of them through a product); dt is checked
// as it is read.
//
// exp(cum_i - cum_j) is factored per 32-row block r of the chunk as
// exp(cum_i - cum_r) * exp(cum_r - cum_j): both factors are at most 1 for
// j before the block, and inside the block the second factor is bounded by
// the block's own dt range, which is checked; a block whose range could
// overflow fp32 computes its diagonal terms one exp at a time.
#include "ssm_internal.cuh"
#include "tc.cuh"
#include "tma.cuh"

namespace ssm {
namespace {

constexpr int Q = 128, SP = 64, SN = 128;
constexpr int kThreads = 256;
constexpr uint32_t kTile128 = 128 * 128;  // one 64-wide (128-byte) column block of a 128-row tile
constexpr uint32_t OFF_C = 0;                      // C  [i][n]  two n blocks: A of C B^T and of Z (K-major);
constexpr uint32_t OFF_M = OFF_C;                  //   then M [i][j], two j blocks: A of Y (K-major)
constexpr uint32_t OFF_B = OFF_C + 2 * kTile128;   // B  [j][n]  B of C B^T (K-major); A of dS^T (MN-major)
constexpr uint32_t OFF_X = OFF_B + 2 * kTile128;   // X  [j][p]  B of Y (MN-major)
constexpr uint32_t OFF_S = OFF_X + kTile128;       // S  [n][p]  B of Z (MN-major);
constexpr uint32_t OFF_XW = OFF_S;                 //   then (w o X) [j][p]: B of dS^T (MN-major)
constexpr uint32_t OFF_MISC = OFF_S + kTile128;
// misc: cum[128], dt[128], colf[4][128], wsum[4], safe[4], mbarriers (MMA, loads), tmem base, gate
constexpr uint32_t M_CUM = 0, M_DT = 512, M_COLF = 1024, M_WSUM = 3072, M_SAFE = 3088, M_BAR = 3104,
                   M_TMEM = 3112, M_GATE = 3116, M_LDBAR = 3120;
constexpr uint32_t kSsdSmem = OFF_MISC + 3200 + 1024;  // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 256;  // [0,128) C B^T, then dS^T in [64,128); Y in [128,192); Z in [192,256)

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
}

// 16-byte chunk c (of 8 bf16) of row r in a 128-byte-row swizzled block.
__device__ __forceinline__ uint32_t chunk_off(uint32_t r, uint32_t c) { return r * 128u + (((c ^ r) & 7u) << 4); }

// K = 128 product into TMEM: 8 MMAs of K = 16.  K-major operands step 32
// bytes along their 128-byte row and 16 KiB to the next 64-wide K block;
// MN-major operands step 16 rows (2 KiB).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int ks) {
    return tc::smem_desc_sw128(base + (uint32_t)(ks >> 2) * kTile128 + (uint32_t)(ks & 3) * 32u, 1024);
}
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int ks) {
    // leading offset: stride between 64-wide MN blocks; stride offset: 8-row K groups
    return tc::smem_desc_sw128_lbo(base + (uint32_t)ks * 2048u, kTile128, 1024);
}

template <typename TI>
__global__ void __launch_bounds__(kThreads, 2)
    scan_ssd_kernel(const __grid_constant__ ScanArgs a, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c) {
    static_assert(sizeof(TI) == 2, "tensor-core scan takes bf16 x, B and C");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);
    unsigned char *misc = smem + OFF_MISC;
    float *s_cum = reinterpret_cast<float *>(misc + M_CUM);
    float *s_dt = reinterpret_cast<float *>(misc + M_DT);
    float *s_colf = reinterpret_cast<float *>(misc + M_COLF);  // [4][128]
    float *s_wsum = reinterpret_cast<float *>(misc + M_WSUM);
    int *s_safe = reinterpret_cast<int *>(misc + M_SAFE);
    uint64_t *s_bar = reinterpret_cast<uint64_t *>(misc + M_BAR);
    uint64_t *s_ldbar = reinterpret_cast<uint64_t *>(misc + M_LDBAR);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(misc + M_TMEM);
    uint32_t *s_gate = reinterpret_cast<uint32_t *>(misc + M_GATE);

    const int h = blockIdx.x, i_seq = blockIdx.y;
    const int t0 = a.cu[i_seq], t1 = a.cu[i_seq + 1];
    if (t1 <= t0) return;  // empty chunk: consumes its sequence number only
    const int slot = a.slots[i_seq];
    const int H = a.H, g = h / a.hpg;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row = tid & 127;      // token row (P1, P3, P5) or state column n
    const int half = tid >> 7;      // which half of the columns this thread takes
    const int rb = (tid >> 5) & 3;  // 32-row block of `row` = this warp's TMEM lane quadrant

    if (tid == 0) {
        uint32_t gate = 0;
        if (a.slot_flags[slot] & kSlotPoisoned) gate = SSM_FLAG_POISONED_SLOT;
        else if (a.check_log && a.log_len[slot] != 0) gate = SSM_FLAG_LOG_NOT_EMPTY;
        *s_gate = gate;
        mbar_init(s_bar, 1);
        mbar_init(s_ldbar, 1);
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
    const uint32_t lane_addr = (uint32_t)(32 * rb) << 16;  // TMEM lane quadrant of this warp

    const float A = a.A[h], D = a.D[h];
    TI *yg = reinterpret_cast<TI *>(a.y);
    float *st = current_state(a.state, a.snap, a.cur, a.n_slots, (size_t)H * SP * SN, (size_t)SP * SN, slot, h);

    // state: thread (n, half) holds S[p][n] for p in [32 half, 32 half + 32)
    const int n_col = row, p0 = 32 * half;
    float S[32];
#pragma unroll
    for (int p = 0; p < 32; ++p) S[p] = st[(size_t)(p0 + p) * SN + n_col];
    auto write_state_copy = [&]() {  // bf16 copy, row n of the [n][p] tile, this half's 4 chunks
#pragma unroll
        for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4 *>(smem + OFF_S + chunk_off(n_col, 4 * half + c)) =
                make_uint4(pack_bf16(S[8 * c + 0], S[8 * c + 1]), pack_bf16(S[8 * c + 2], S[8 * c + 3]),
                           pack_bf16(S[8 * c + 4], S[8 * c + 5]), pack_bf16(S[8 * c + 6], S[8 * c + 7]));
    };
    write_state_copy();

    constexpr uint32_t kIdCB = tc::idesc_bf16_f32(128, 128);                 // K-major x K-major
    constexpr uint32_t kIdY = tc::idesc_bf16_f32(128, 64) | (1u << 16);      // B MN-major
    constexpr uint32_t kIdZ = tc::idesc_bf16_f32(128, 64) | (1u << 16);      // B MN-major
    constexpr uint32_t kIdDS = tc::idesc_bf16_f32(128, 64) | (1u << 15) | (1u << 16);  // both MN-major
    uint32_t phase = 0, ld_phase = 0;
    // The chunk's tiles, one load phase per chunk: C and B (4 boxes) once the previous chunk's
    // MMAs have read them, x (1 box) once its outputs are written.
    auto load_cb = [&](int ty) {
        mbar_arrive_expect_tx(s_ldbar, 5u * kTile128);
        tma_load_2d(smem + OFF_C, &tm_c, g * SN, ty, s_ldbar);
        tma_load_2d(smem + OFF_C + kTile128, &tm_c, g * SN + 64, ty, s_ldbar);
        tma_load_2d(smem + OFF_B, &tm_b, g * SN, ty, s_ldbar);
        tma_load_2d(smem + OFF_B + kTile128, &tm_b, g * SN + 64, ty, s_ldbar);
    };
    auto load_x = [&](int ty) { tma_load_2d(smem + OFF_X, &tm_x, h * SP, ty, s_ldbar); };
    bool bad = false, timeout = false;
    const int L = t1 - t0;
    // dt of this thread's row, one chunk ahead (a strided load, kept off the chunk's critical path)
    float dt_next = 0.f;
    if (half == 1 && row < (L < Q ? L : Q)) dt_next = load_dt(a.dt, (size_t)(t0 + row) * H + h, a.dt_bf16);
    if (tid == 0) {
        load_cb(t0);
        load_x(t0);
    }
    for (int c0 = 0; c0 < L; c0 += Q) {
        const int len = L - c0 < Q ? L - c0 : Q;
        const bool valid = row < len;
        const size_t tok = (size_t)(t0 + c0 + row);

        // ---- P1: the chunk's rows of C, B (two 64-column boxes each) and x, issued by TMA into
        // the swizzled tiles (the layout chunk_off describes) as soon as the previous chunk was
        // done with each tile; dt prefix sums while they land
        float dtv = 0.f;
        if (half == 1) {
            dtv = dt_next;
            bad |= !isfinite(dtv);
            // inclusive prefix sum over the 128 rows (warps 4..7)
            float v = dtv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (lane == 31) s_wsum[rb] = v;
            s_dt[row] = dtv;
            bar_sync_named(1, 128);
            for (int w = 0; w < rb; ++w) v += s_wsum[w];
            s_cum[row] = A * v;
        }
        if (__syncthreads_or(!mbar_wait(s_ldbar, ld_phase & 1u))) {  // uniform across the CTA
            timeout = true;
            break;
        }
        ++ld_phase;
        if (!valid) {  // rows past the sequence: the boxes hold the next tokens of the tensor, or zeros
            if (half == 0) {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint32_t off = (uint32_t)(c >> 3) * kTile128 + chunk_off((uint32_t)row, (uint32_t)c);
                    *reinterpret_cast<uint4 *>(smem + OFF_C + off) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(smem + OFF_B + off) = make_uint4(0, 0, 0, 0);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(smem + OFF_X + chunk_off((uint32_t)row, (uint32_t)c)) = make_uint4(0, 0, 0, 0);
            }
        }
        const float cum_last = s_cum[Q - 1];
        const float cum = s_cum[row];
        // column factors colf[r][j] = exp(cum_{32r} - cum_j) dt_j for j < 32 r + 32,
        // and whether block r's own range keeps them finite
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int r = 2 * half + q;
            const float ref = s_cum[32 * r];
            s_colf[r * Q + row] = row < 32 * r + 32 ? expf(ref - cum) * s_dt[row] : 0.f;
        }
        if (tid < 4) s_safe[tid] = (s_cum[32 * tid] - s_cum[32 * tid + 31]) < 80.f;
        tc::fence_proxy_async_smem();
        __syncthreads();

        if (half == 1) {  // dt of the next chunk, while this one is on the tensor cores
            const int c1 = c0 + Q, len1 = L - c1 < Q ? L - c1 : Q;
            dt_next = row < len1 ? load_dt(a.dt, (size_t)(t0 + c1 + row) * H + h, a.dt_bf16) : 0.f;
        }

        // ---- P2: C B^T and Z = C S^T (S before the chunk); after them C and S are free
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                tc::mma_bf16(tmem, kmajor_desc(sbase + OFF_C, ks), kmajor_desc(sbase + OFF_B, ks), kIdCB, ks > 0);
                tc::mma_bf16(tmem + 192, kmajor_desc(sbase + OFF_C, ks), mnmajor_desc(sbase + OFF_S, ks), kIdZ, ks > 0);
            }
            tc::mma_commit(s_bar);
        }

        if (__syncthreads_or(!mbar_wait(s_bar, phase & 1u))) {  // uniform across the CTA
            timeout = true;
            break;
        }
        ++phase;
        tc::fence_after_sync();

        // ---- P3: M = C B^T o decay o dt, masked to j <= i (row i = row, columns of this half).
        // A warp's rows lie in one 32-row block rb, so each 32-column block jb is, for the whole
        // warp, either right of the diagonal (all zero), left of it (erow x colf, no mask) or the
        // diagonal block itself (masked; exact exps where the block's range is not safe).
        {
            const int i = row;
            const float erow = expf(cum - s_cum[32 * rb]);  // <= 1
            const bool safe = s_safe[rb] != 0;
            const float *colf = s_colf + rb * Q;
#pragma unroll 1
            for (int jb = 64 * half; jb < 64 * half + 64; jb += 32) {
                uint4 *mrow = reinterpret_cast<uint4 *>(smem + OFF_M + (uint32_t)(jb >> 6) * kTile128);
                const uint32_t c0q = (uint32_t)(jb & 63) >> 3;  // first 8-column chunk of the block
                if (jb > 32 * rb) {  // right of the diagonal
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8)
                        *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(mrow) +
                                                   chunk_off((uint32_t)i, c0q + q8)) = make_uint4(0, 0, 0, 0);
                    continue;
                }
                float cb[32];
                tc::tmem_ld32(tmem + lane_addr + (uint32_t)jb, cb);
                const bool plain = jb < 32 * rb || safe, diag = jb == 32 * rb;
                const float4 *c4 = reinterpret_cast<const float4 *>(colf + jb);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {  // 8 columns at a time
                    float f[8];
                    if (plain) {
                        const float4 ca = c4[2 * q8], cc = c4[2 * q8 + 1];
                        f[0] = erow * ca.x; f[1] = erow * ca.y; f[2] = erow * ca.z; f[3] = erow * ca.w;
                        f[4] = erow * cc.x; f[5] = erow * cc.y; f[6] = erow * cc.z; f[7] = erow * cc.w;
                    } else {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int j = jb + 8 * q8 + u;
                            f[u] = expf(cum - s_cum[j]) * s_dt[j];
                        }
                    }
                    if (diag) {  // the diagonal block: j <= i only
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (jb + 8 * q8 + u > i) f[u] = 0.f;
                    }
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int u = 8 * q8 + 2 * e;
                        pk[e] = pack_bf16(cb[u] * f[2 * e], cb[u + 1] * f[2 * e + 1]);
                    }
                    *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(mrow) + chunk_off((uint32_t)i, c0q + q8)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
            // w o X, row j = row, this half's 4 chunks: weight of token j in the state update
            const float wt = expf(cum_last - cum) * s_dt[row];
#pragma unroll
            for (int c = 4 * half; c < 4 * half + 4; ++c) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(smem + OFF_X + chunk_off((uint32_t)row, (uint32_t)c));
                const float2 f0 = unpack_bf16(xv.x), f1 = unpack_bf16(xv.y);
                const float2 f2 = unpack_bf16(xv.z), f3 = unpack_bf16(xv.w);
                *reinterpret_cast<uint4 *>(smem + OFF_XW + chunk_off((uint32_t)row, (uint32_t)c)) =
                    make_uint4(pack_bf16(f0.x * wt, f0.y * wt), pack_bf16(f1.x * wt, f1.y * wt),
                               pack_bf16(f2.x * wt, f2.y * wt), pack_bf16(f3.x * wt, f3.y * wt));
            }
        }
        tc::fence_before_sync();
        tc::fence_proxy_async_smem();
        __syncthreads();

        // ---- P4: Y = M X, dS^T = B^T (w o X)
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                tc::mma_bf16(tmem + 128, kmajor_desc(sbase + OFF_M, ks), mnmajor_desc(sbase + OFF_X, ks), kIdY, ks > 0);
                tc::mma_bf16(tmem + 64, mnmajor_desc(sbase + OFF_B, ks), mnmajor_desc(sbase + OFF_XW, ks), kIdDS, ks > 0);
            }
            tc::mma_commit(s_bar);
        }
        if (__syncthreads_or(!mbar_wait(s_bar, phase & 1u))) {
            timeout = true;
            break;
        }
        ++phase;
        tc::fence_after_sync();

        if (tid == 0 && c0 + Q < L) load_cb(t0 + c0 + Q);  // C (now M) and B are read

        // ---- P5: outputs of row i (this half's 32 columns p), state update of column n = row,
        // 16 columns at a time
        {
            const float ecum = expf(cum);
            const float dA = expf(cum_last);
            // Non-finite inputs show here: every x, B and C value reaches y or the state
            // increment through a product (a NaN or Inf times anything, zero included, is not
            // finite), so v * 0 summed over them is NaN exactly when one of them is not finite.
            float nf = 0.f;
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                float yv[16], zv[16];
                tc::tmem_ld16(tmem + lane_addr + 128u + (uint32_t)(p0 + 16 * hc), yv);
                tc::tmem_ld16(tmem + lane_addr + 192u + (uint32_t)(p0 + 16 * hc), zv);
                uint4 outc[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint4 xc = *reinterpret_cast<const uint4 *>(
                        smem + OFF_X + chunk_off((uint32_t)row, (uint32_t)(4 * half + 2 * hc + c)));
                    const uint32_t xw4[4] = {xc.x, xc.y, xc.z, xc.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 xf = unpack_bf16(xw4[e]);
                        const int q = 8 * c + 2 * e;
                        const float v0 = fmaf(ecum, zv[q], yv[q]) + D * xf.x, v1 = fmaf(ecum, zv[q + 1], yv[q + 1]) + D * xf.y;
                        nf = fmaf(v0, 0.f, fmaf(v1, 0.f, nf));
                        o[e] = pack_bf16(v0, v1);
                    }
                    outc[c] = make_uint4(o[0], o[1], o[2], o[3]);
                }
                if (valid) {
                    uint4 *yo = reinterpret_cast<uint4 *>(yg + (tok * H + h) * SP + p0 + 16 * hc);
                    yo[0] = outc[0];
                    yo[1] = outc[1];
                }
            }
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                float ds[16];
                tc::tmem_ld16(tmem + lane_addr + 64u + (uint32_t)(p0 + 16 * hc), ds);
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    nf = fmaf(ds[p], 0.f, nf);
                    S[16 * hc + p] = fmaf(dA, S[16 * hc + p], ds[p]);
                }
            }
            bad |= nf != nf;
        }
        write_state_copy();
        tc::fence_before_sync();
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && c0 + Q < L) load_x(t0 + c0 + Q);  // x is read
    }

    const bool any_bad = __syncthreads_or(bad);
    if (!any_bad && !timeout) {
#pragma unroll
        for (int p = 0; p < 32; ++p) st[(size_t)(p0 + p) * SN + n_col] = S[p];
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
    const TensorMapEncode enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    // tokens of this launch as rows: x [T][H * P], B and C [T][G * N]; 64-column x 128-row boxes,
    // 128-byte swizzle, zeros past the last token
    const cuuint64_t T = (cuuint64_t)a.cu[a.n_seq];
    const cuuint32_t box[2] = {64u, (cuuint32_t)Q};
    const cuuint32_t es[2] = {1u, 1u};
    CUtensorMap mx, mb, mc;
    const cuuint64_t xd[2] = {(cuuint64_t)a.H * SP, T}, xs[1] = {(cuuint64_t)a.H * SP * 2};
    const cuuint64_t bd[2] = {(cuuint64_t)a.G * SN, T}, bs[1] = {(cuuint64_t)a.G * SN * 2};
    const auto encode = [&](CUtensorMap *m, const void *base, const cuuint64_t *d, const cuuint64_t *st) {
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), d, st, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (!encode(&mx, a.x, xd, xs) || !encode(&mb, a.B, bd, bs) || !encode(&mc, a.C, bd, bs))
        return cudaErrorNotSupported;
    auto k = scan_ssd_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSsdSmem);
    if (e != cudaSuccess) return e;
    k<<<dim3(a.H, a.n_seq), kThreads, kSsdSmem, s>>>(a, mx, mb, mc);
    return cudaGetLastError();
}

}  // namespace ssm
