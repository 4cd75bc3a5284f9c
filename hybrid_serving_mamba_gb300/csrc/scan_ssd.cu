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
//   dS^T    = B^T (w o X)     w_j = exp(cum_last - cum_j) dt_j, w o X as bf16 hi + lo
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
constexpr uint32_t OFF_XW = OFF_S;                 //   then (w o X)_hi [j][p]: B of dS^T (MN-major)
constexpr uint32_t OFF_XWLO = OFF_M;               // (w o X)_lo [j][p] in M's first block, once Y has read M
constexpr uint32_t OFF_MISC = OFF_S + kTile128;
// misc: cum[128], dt[128], colf[4][128], wsum[4], safe[4], mbarriers (MMA, loads), tmem base, gate
constexpr uint32_t M_CUM = 0, M_DT = 512, M_COLF = 1024, M_WSUM = 3072, M_SAFE = 3088, M_BAR = 3104,
                   M_TMEM = 3112, M_GATE = 3116, M_LDBAR = 3120, M_CMAX = 3136, M_CMIN = 3152;
// the factored form is taken while exp(+-kFactorRange) stays far inside fp32 (max about exp(88))
constexpr float kFactorRange = 70.f;
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
    float *s_cmax = reinterpret_cast<float *>(misc + M_CMAX);  // [4] per row block
    float *s_cmin = reinterpret_cast<float *>(misc + M_CMIN);  // [4]

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
    // bf16 copy of sc * S, row n of the [n][p] tile, this half's 4 chunks (the B operand of Z)
    auto write_state_copy = [&](float sc) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4 *>(smem + OFF_S + chunk_off(n_col, 4 * half + c)) =
                make_uint4(pack_bf16(sc * S[8 * c + 0], sc * S[8 * c + 1]), pack_bf16(sc * S[8 * c + 2], sc * S[8 * c + 3]),
                           pack_bf16(sc * S[8 * c + 4], sc * S[8 * c + 5]), pack_bf16(sc * S[8 * c + 6], sc * S[8 * c + 7]));
    };

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

    // One chunk's dt (rows: warps 4..7): prefix sums cum_i = A (dt_0 + .. + dt_i), and the range of
    // cum, from which every thread takes the chunk's reference point and whether the factored form
    // below is safe for it.  Called by every thread.
    auto chunk_setup = [&](float dtv) {
        if (half == 1) {
            bad |= !isfinite(dtv);
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
            const float c = A * v;
            s_cum[row] = c;
            float mx = c, mn = c;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            }
            if (lane == 0) {
                s_cmax[rb] = mx;
                s_cmin[rb] = mn;
            }
        }
        __syncthreads();
    };
    // The factored form: exp(cum_i - cum_j) = exp(cum_i - ref) exp(ref - cum_j) with ref = cum at the
    // middle row of the chunk, so that the decay-masked product is a plain causal mask of C B^T,
    // shared by every row's scale.  Safe while both factors, and exp(ref) that scales the state copy,
    // stay far inside fp32 (a NaN range is not safe either: the exact path finds the NaN).
    auto fast_ok = [&](int len, float &ref_out) -> bool {
        const float ref = s_cum[(len - 1) >> 1];
        const float mx = fmaxf(fmaxf(s_cmax[0], s_cmax[1]), fmaxf(s_cmax[2], s_cmax[3]));
        const float mn = fminf(fminf(s_cmin[0], s_cmin[1]), fminf(s_cmin[2], s_cmin[3]));
        ref_out = ref;
        return (mx - ref <= kFactorRange) && (ref - mn <= kFactorRange) && (ref >= -kFactorRange);
    };

    // chunk 0: its dt, its form, the state copy its Z reads, its tiles
    float ref = 0.f;
    bool fast;
    {
        const float d0 = (half == 1 && row < (L < Q ? L : Q)) ? load_dt(a.dt, (size_t)(t0 + row) * H + h, a.dt_bf16)
                                                             : 0.f;
        chunk_setup(d0);
        fast = fast_ok(L < Q ? L : Q, ref);
        write_state_copy(fast ? expf(ref) : 1.f);
    }
    float dt_next = 0.f;
    if (tid == 0) {
        load_cb(t0);
        load_x(t0);
    }
    for (int c0 = 0; c0 < L; c0 += Q) {
        const int len = L - c0 < Q ? L - c0 : Q;
        const bool valid = row < len;
        const size_t tok = (size_t)(t0 + c0 + row);

        // ---- P1: dt of the next chunk (a strided load, off the critical path); the chunk's rows
        // of C, B (two 64-column boxes each) and x, issued by TMA into the swizzled tiles as soon as
        // the previous chunk was done with each tile
        const int c1 = c0 + Q, len1 = L - c1 < Q ? L - c1 : Q;
        if (half == 1) dt_next = row < len1 ? load_dt(a.dt, (size_t)(t0 + c1 + row) * H + h, a.dt_bf16) : 0.f;
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
        const float dtr = s_dt[row];
        if (!fast) {
            // exact form: column factors colf[r][j] = exp(cum_{32r} - cum_j) dt_j for j < 32 r + 32,
            // and whether block r's own range keeps them finite
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int r = 2 * half + q;
                const float rf = s_cum[32 * r];
                s_colf[r * Q + row] = row < 32 * r + 32 ? expf(rf - cum) * dtr : 0.f;
            }
            if (tid < 4) s_safe[tid] = (s_cum[32 * tid] - s_cum[32 * tid + 31]) < 80.f;
        }
        tc::fence_proxy_async_smem();
        __syncthreads();

        // ---- P2: C B^T and Z = C (sc S)^T (S before the chunk; sc = exp(ref) in the factored form,
        // whose Z shares the accumulator of Y); after them C and the state copy are free
        const uint32_t zcol = fast ? 128u : 192u;
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                tc::mma_bf16(tmem, kmajor_desc(sbase + OFF_C, ks), kmajor_desc(sbase + OFF_B, ks), kIdCB, ks > 0);
                tc::mma_bf16(tmem + zcol, kmajor_desc(sbase + OFF_C, ks), mnmajor_desc(sbase + OFF_S, ks), kIdZ, ks > 0);
            }
            tc::mma_commit(s_bar);
        }

        if (__syncthreads_or(!mbar_wait(s_bar, phase & 1u))) {  // uniform across the CTA
            timeout = true;
            break;
        }
        ++phase;
        tc::fence_after_sync();

        uint4 xw_lo[4];  // this thread's lo half of the state operand, row `row`, chunks 4 half .. 4 half + 3
        // ---- P3: the causal product operand (row i = row, columns of this half) and the state
        // operand.  A warp's rows lie in one 32-row block rb, so each 32-column block jb is, for the
        // whole warp, either right of the diagonal (all zero), left of it (no mask) or the diagonal
        // block itself (masked to j <= i).
        //   factored:  L[i][j] = C B^T[i][j] (j <= i);  X~_j = exp(ref - cum_j) dt_j x_j
        //   exact:     M[i][j] = C B^T[i][j] exp(cum_i - cum_j) dt_j (j <= i);  (w o X)_j = exp(cum_last - cum_j) dt_j x_j
        {
            const int i = row;
            const float erow = fast ? 1.f : expf(cum - s_cum[32 * rb]);  // <= 1
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
                const bool diag = jb == 32 * rb;
                if (fast) {
#pragma unroll
                    for (int q8 = 0; q8 < 4; ++q8) {
                        float f[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) f[u] = (diag && jb + 8 * q8 + u > i) ? 0.f : cb[8 * q8 + u];
                        *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(mrow) +
                                                   chunk_off((uint32_t)i, c0q + q8)) =
                            make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                                       pack_bf16(f[6], f[7]));
                    }
                    continue;
                }
                const bool plain = jb < 32 * rb || safe;
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
            // the state operand, row j = row, this half's 4 chunks, as hi (to the tile now) and lo
            // (kept for the second product)
            const float wt = (fast ? expf(ref - cum) : expf(cum_last - cum)) * dtr;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 xv =
                    *reinterpret_cast<const uint4 *>(smem + OFF_X + chunk_off((uint32_t)row, (uint32_t)(4 * half + c)));
                const uint32_t xw4[4] = {xv.x, xv.y, xv.z, xv.w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack_bf16(xw4[e]);
                    const float v0 = f.x * wt, v1 = f.y * wt;
                    hi[e] = pack_bf16(v0, v1);
                    const float2 hf = unpack_bf16(hi[e]);
                    lo[e] = pack_bf16(v0 - hf.x, v1 - hf.y);
                }
                *reinterpret_cast<uint4 *>(smem + OFF_XW + chunk_off((uint32_t)row, (uint32_t)(4 * half + c))) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
                xw_lo[c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        tc::fence_before_sync();
        tc::fence_proxy_async_smem();
        __syncthreads();

        // ---- P4: factored: Y~ = L X~_hi into Z's accumulator; exact: Y = M X.  dS^T = B^T (hi operand)
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                if (fast)
                    tc::mma_bf16(tmem + 128, kmajor_desc(sbase + OFF_M, ks), mnmajor_desc(sbase + OFF_XW, ks), kIdY, true);
                else
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
        // ---- P4b: with M / L read, the lo operand into its tile and dS^T += B^T (lo operand); waited
        // for only before the state update, so it runs under the outputs below
#pragma unroll
        for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4 *>(smem + OFF_XWLO + chunk_off((uint32_t)row, (uint32_t)(4 * half + c))) = xw_lo[c];
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                tc::mma_bf16(tmem + 64, mnmajor_desc(sbase + OFF_B, ks), mnmajor_desc(sbase + OFF_XWLO, ks), kIdDS, true);
            tc::mma_commit(s_bar);
        }
        tc::fence_after_sync();

        // ---- P5: outputs of row i (this half's 32 columns p), 16 columns at a time
        //   factored: y_i = exp(cum_i - ref) (Z~ + Y~)_i + D x_i;  exact: y_i = Y_i + exp(cum_i) Z_i + D x_i
        // Non-finite inputs show here and in the state increment: every x, B and C value reaches one
        // of them through a product (a NaN or Inf times anything, zero included, is not finite), so
        // v * 0 summed over them is NaN exactly when one of them is not finite.
        float nf = 0.f;
        {
            const float rs = fast ? expf(cum - ref) : 1.f;
            const float ecum = fast ? 0.f : expf(cum);
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                float yv[16], zv[16];
                tc::tmem_ld16(tmem + lane_addr + 128u + (uint32_t)(p0 + 16 * hc), yv);
                if (!fast) tc::tmem_ld16(tmem + lane_addr + 192u + (uint32_t)(p0 + 16 * hc), zv);
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
                        float v0, v1;
                        if (fast) {
                            v0 = fmaf(rs, yv[q], D * xf.x);
                            v1 = fmaf(rs, yv[q + 1], D * xf.y);
                        } else {
                            v0 = fmaf(ecum, zv[q], yv[q]) + D * xf.x;
                            v1 = fmaf(ecum, zv[q + 1], yv[q + 1]) + D * xf.y;
                        }
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
        }
        // this chunk's state factors, then the next chunk's dt, form and reference point (every
        // thread is done with this chunk's cum)
        const float dA = expf(cum_last);
        const float cds = fast ? expf(cum_last - ref) : 1.f;
        bool fast_next = fast;
        float ref_next = ref;
        __syncthreads();
        if (len1 > 0) {
            chunk_setup(dt_next);
            fast_next = fast_ok(len1, ref_next);
        }
        // the state increment (both products), then C and B of the next chunk may land
        if (__syncthreads_or(!mbar_wait(s_bar, phase & 1u))) {
            timeout = true;
            break;
        }
        ++phase;
        tc::fence_after_sync();
        if (tid == 0 && len1 > 0) load_cb(t0 + c1);
        // ---- state update of column n = row: S <- exp(cum_last) S + cds dS, 16 columns at a time
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            float ds[16];
            tc::tmem_ld16(tmem + lane_addr + 64u + (uint32_t)(p0 + 16 * hc), ds);
#pragma unroll
            for (int p = 0; p < 16; ++p) {
                nf = fmaf(ds[p], 0.f, nf);
                S[16 * hc + p] = fmaf(dA, S[16 * hc + p], cds * ds[p]);
            }
        }
        bad |= nf != nf;
        if (len1 > 0) write_state_copy(fast_next ? expf(ref_next) : 1.f);
        fast = fast_next;
        ref = ref_next;
        tc::fence_before_sync();
        tc::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && len1 > 0) load_x(t0 + c1);  // x is read
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

cudaError_t launch_scan_ssd(const Pool &pool, const ScanArgs &a, cudaStream_t s, const char **path) {
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
    if (path) *path = "scan_ssd";
    return cudaGetLastError();
}

}  // namespace ssm
