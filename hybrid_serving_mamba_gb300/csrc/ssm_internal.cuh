// Internal declarations of libssmstate (not part of the C ABI).
//
// Thread layout shared by the state-streaming kernels (decode, copy verify,
// replay verify, fold, sequential scan): one CTA per (request or sequence,
// head).  A head's state is P rows of N fp32 values, N contiguous.  Each row
// is covered by LPR = N / 16 lanes; a lane owns 16 values of the row as four
// float4 at float4 indices sub, sub + LPR, sub + 2 LPR, sub + 3 LPR, so each
// 128-bit load or store instruction of a warp touches 32 / LPR rows in
// contiguous 16 * LPR-byte runs (fully used 128-byte lines for N >= 128).
// A thread owns kRowsPerThread rows; a warp covers RPW * kRowsPerThread rows,
// RPW = 32 / LPR, and the CTA has ceil(P / (RPW * kRowsPerThread)) warps.
// C . h over a row is a partial dot over the lane's 16 values followed by an
// xor-shuffle reduction over the LPR lanes of the row.
#pragma once

#include <cuda.h>  // CUtensorMap (the encoder is looked up at run time)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <vector>

#include "ssm_state.h"

namespace ssm {

constexpr int kMaxSlotsPerLaunch = 1024;  // slot lists travel in kernel parameters
constexpr int kMaxSeqPerLaunch = 1024;
constexpr int kRowsPerThread = 2;
constexpr int kMaxThreads = 512;  // per CTA of the state-streaming kernels
constexpr uint32_t kSlotPoisoned = 1u;
constexpr int kMaxFoldK = 64;  // largest K extent (log capacity rounded up to 16) of the tensor-core fold

// ---------------------------------------------------------------- pool

struct Pool {
    ssm_config cfg;
    int n_slots = 0;
    int device = 0;
    int H = 0, P = 0, N = 0, G = 0, hpg = 0;
    size_t pn = 0;    // P * N floats per head
    size_t hpn = 0;   // H * P * N floats per slot
    int t1max = 0;    // max tokens per verify step
    int wcap = 0;     // replay log capacity: W - 1 + t1max (W - 1 + 2 t1max when the verify folds)
    int wwin = 0;     // replay: longest window a verify replays, W - 1 + t1max
    bool fold_in_verify = false;  // SSM_FOLD_IN_VERIFY
    size_t in_bytes = 0;  // bytes per x / B / C element

    float *state = nullptr;      // [n_slots][H][P][N]
    float *snap = nullptr;       // copy mode: [2][t1max][n_slots][H][P][N]
    void *log_x = nullptr;       // replay: [n_slots][wcap][H][P]   input dtype
    float *log_dt = nullptr;     // replay: [n_slots][wcap][H]
    void *log_B = nullptr;       // replay: [n_slots][wcap][G][N]   input dtype
    int64_t *d_position = nullptr;
    int32_t *d_log_len = nullptr;
    int32_t *d_cur = nullptr;          // copy mode: -1 = base state, else half * t1max + j
    uint32_t *d_slot_flags = nullptr;  // kSlotPoisoned
    uint32_t *d_flags = nullptr;       // sticky SSM_FLAG_* bits
    float *d_stage = nullptr;          // one slot's state, for checkpoint / restore
    // replay scratch: C_j . B_s of one launch's requests, [cb_rows][G][t1max][wcap]
    float *d_cb = nullptr;
    int cb_rows = 0;
    int cb_w = 0;                      // row stride of d_cb: wwin rounded up to 4 floats
    float *d_wsc = nullptr;            // replay: W[j][s] per head, [cb_rows][H][t1max][cb_w]
    float *d_dec = nullptr;            // replay: decay_j per head, [cb_rows][H][t1pad]
    float *d_cf = nullptr;             // replay: C_j in fp32 per group, [cb_rows][G][cf_rows][N]
    int cf_rows = 0;                   // t1max rounded up to 16
    int t1pad = 0;                     // t1max rounded up to 4
    CUtensorMap tm_state;              // replay: checkpoint rows, 32-column boxes, 128-byte swizzle
    CUtensorMap tm_logx;               // replay: one head's log of x rows per box
    bool tm_ok = false;                // both maps encoded
    CUtensorMap tm_state2;             // replay, tensor cores: 32 columns x 128 rows (two heads) per box
    CUtensorMap tm_logx2;              // replay, tensor cores: two heads' logs of x rows per box
    bool tm_tc_ok = false;             // the two maps above encoded
    CUtensorMap tm_logB;               // replay, bf16, N = 128: fold_kp logged B rows x 64 columns of a group per box
    bool tm_fold_ok = false;           // tm_state2, tm_logx2 and tm_logB encoded for the tensor-core fold
    int fold_kp = 0;                   // K extent of the tensor-core fold (32, 48 or 64 >= the longest window)
    int2 *d_fold_items = nullptr;      // (request index, tokens to fold) of one commit launch
    int32_t *d_fold_count = nullptr;
    // fold in verify: where each slot's last verify staged its tokens; the verify's request lists
    // (plain requests; (request, log length) of the requests whose full log it folds) and, for the
    // commit, (request, from, to, count) of staged tokens to move to the end of the log
    int32_t *d_stage_pos = nullptr;    // [n_slots]
    int32_t *d_plain = nullptr;        // [kMaxSlotsPerLaunch]
    int2 *d_fv_items = nullptr;        // [kMaxSlotsPerLaunch]
    int4 *d_moves = nullptr;           // [kMaxSlotsPerLaunch]
    int32_t *d_counts = nullptr;       // plain, fold-in-verify, moves
    CUtensorMap tm_logx_fv;            // both heads' whole logs (wcap rows) per box
    int sm_count = 1;
    size_t bytes = 0;

    // host-buffer decode: two staging sets, each x | dt | B | C | y of one step, and the copy streams
    struct HostPipe {
        cudaStream_t up = nullptr, down = nullptr;
        // start; then per set: inputs landed, inputs consumed, output written, output read back
        cudaEvent_t start = nullptr, in_ready[2] = {}, used[2] = {}, y_ready[2] = {}, y_free[2] = {};
        char *buf = nullptr;  // [2][set_cap]
        size_t set_cap = 0;
    } hpipe;

    // host mirror
    std::vector<int64_t> next_chunk, epoch;
    std::vector<uint8_t> released;
    std::vector<int32_t> pending_ntok;  // n_tok of the last uncommitted verify, 0 = none
    const char *last_path = "none";
    int test_stall = 0;  // ssm_debug_stall_next_verify, one-shot
};

// ---------------------------------------------------------------- kernel args

struct StepArgs {  // decode, copy verify, replay verify
    const void *x, *dt, *B, *C;
    const float *A, *D;
    void *y;
    float *state;
    float *snap;
    void *log_x;
    float *log_dt;
    void *log_B;
    float *cb;        // replay scratch (see Pool::d_cb)
    int cb_w;         // its row stride in floats (a multiple of 4)
    float *wsc;       // replay scratch (see Pool::d_wsc); null: no tensor-map verify
    float *dec;
    float *cf;
    int t1pad;
    int cf_rows;      // row stride of a (request, group) block of cf, in rows of N
    int cf_nm;        // 0: cf rows plain; else NM rows (T1 padded with zero rows) as the MMA's K-major
                      // swizzled operand: [column block][row][32], 16-byte chunk c of row j at c ^ (j % 8)
    int64_t *position;
    int32_t *log_len;
    int32_t *cur;
    uint32_t *slot_flags;
    uint32_t *flags;
    int H, P, N, G, hpg;
    int n_slots, t1max, wcap;
    int n_tok;        // tokens per request in this call (1 for decode)
    int dt_bf16;      // dt dtype is bf16
    int check_log;    // replay pool: in-place updates need an empty log
    int wwin;         // replay: longest window (rows of the log boxes the tensor-core kernels load)
    int fold_w;       // fold in verify: W (a log of at least W tokens is folded by this verify); 0: off
    int32_t *stage_pos;   // fold in verify: see Pool
    int32_t *plain;
    int2 *fv_items;
    int32_t *counts;
    int test_stall;   // tests of the failure path: withhold one per-item load (see ssm_debug_stall_next_verify)
    int batch;
    int32_t slots[kMaxSlotsPerLaunch];
};

struct CommitArgs {
    const int32_t *accept;
    const float *A;
    float *state;
    void *log_x;
    float *log_dt;
    void *log_B;
    int64_t *position;
    int32_t *log_len;
    int32_t *cur;
    uint32_t *slot_flags;
    uint32_t *flags;
    int2 *fold_items;
    int32_t *fold_count;
    int H, P, N, G, hpg;
    int n_slots, t1max, wcap, W;
    int fold_grid;    // CTAs of the persistent fold kernel
    int force_fold;
    int flush;        // fold the log only (checkpoint); accept is ignored
    int wwin;         // longest window (rows of the log boxes the tensor-core fold loads)
    int fold_w;       // fold in verify: W; the commit appends unless forced, moving staged tokens first
    int32_t *stage_pos;
    int4 *moves;
    int32_t *counts;
    int batch;
    int32_t slots[kMaxSlotsPerLaunch];
    int32_t ntok[kMaxSlotsPerLaunch];
};

struct ScanArgs {
    const void *x, *dt, *B, *C;
    const float *A, *D;
    void *y;
    float *state;
    float *snap;
    int32_t *cur;
    int n_slots;
    int64_t *position;
    int32_t *log_len;
    uint32_t *slot_flags;
    uint32_t *flags;
    int H, P, N, G, hpg;
    int dt_bf16;
    int check_log;
    int n_seq;
    int32_t cu[kMaxSeqPerLaunch + 1];
    int32_t slots[kMaxSeqPerLaunch];
};

// cuTensorMapEncodeTiled, looked up through the runtime's driver entry point
// once per process; nullptr where the driver does not offer it.
using TensorMapEncode = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);
TensorMapEncode tensor_map_encoder();

// ---------------------------------------------------------------- launchers
// Each returns cudaGetLastError() of its launch(es).

cudaError_t launch_decode(const Pool &pool, const StepArgs &a, cudaStream_t s);
cudaError_t launch_verify_copy(const Pool &pool, const StepArgs &a, cudaStream_t s);
// Replay verify: the C.B prep kernel, then the pipelined kernel where the
// shapes and pointers allow bulk copies, else the one-CTA-per-head kernel.
// *path (if given) names the verify kernel used.
cudaError_t launch_verify_replay(const Pool &pool, const StepArgs &a, cudaStream_t s, const char **path = nullptr);
// Replay verify with the checkpoint streamed by tensor-map copies
// (per-group coefficient kernel + persistent streaming kernel; needs the
// wsc / dec / cf scratch and the pool's tensor maps); cudaErrorNotSupported
// when it cannot run.  replay_tma_encode fills Pool::tm_* (false: shape not
// covered or no encoder in the driver).
cudaError_t launch_verify_replay_tma(const Pool &pool, const StepArgs &a, cudaStream_t s, const char **path);
size_t replay_coef_smem_bytes(const Pool &pool, int n_tok);
bool replay_tma_encode(Pool &p);
// Pipelined replay verify (persistent CTAs, bulk-copy ring); returns
// cudaErrorNotSupported when the shapes or pointers do not allow it.
cudaError_t launch_verify_replay_pipe(const Pool &pool, const StepArgs &a, cudaStream_t s);
// The commit; *path names the fold kernel that ran (or "commit_copy").
cudaError_t launch_commit(const Pool &pool, const CommitArgs &a, cudaStream_t s, const char **path = nullptr);
// The fold on the tensor cores (bf16 pools, P = 64, N = 128, log capacity <= 64);
// cudaErrorNotSupported for other pools.
cudaError_t launch_fold_tc(const Pool &pool, const CommitArgs &a, cudaStream_t s);
// Fold in verify: the requests the coefficient kernel listed as holding a
// full log (StepArgs::fv_items) get the log folded into the checkpoint and
// the step's outputs from the new checkpoint, in one checkpoint read and one
// write (fold_verify.cu).  cudaErrorNotSupported when it cannot run.
cudaError_t launch_fold_verify_tc(const Pool &pool, const StepArgs &a, int NM, cudaStream_t s);
bool fold_verify_fits(const Pool &pool);
// Pipelined fold of the requests the commit listed; cudaErrorNotSupported
// when the shapes or pointers do not allow bulk copies.
cudaError_t launch_fold_pipe(const Pool &pool, const CommitArgs &a, cudaStream_t s);
cudaError_t launch_scan_seq(const Pool &pool, const ScanArgs &a, cudaStream_t s);
// Tensor-core chunked scan (bf16 x / B / C, headdim 64, dstate 128).
bool scan_ssd_supported(const Pool &pool);
// *path names the kernel ("scan_ssd").
cudaError_t launch_scan_ssd(const Pool &pool, const ScanArgs &a, cudaStream_t s, const char **path);
cudaError_t launch_reset(const Pool &pool, const int32_t *slots, int n, cudaStream_t s);
cudaError_t launch_gather(const Pool &pool, const int32_t *slots, int n, float *dst, cudaStream_t s);

// Kernel path of the calling thread's last ssm_verify_replay_static call.
const char *static_last_path();

size_t replay_smem_bytes(const Pool &pool, int n_tok);
size_t replay_prep_smem_bytes(const Pool &pool, int n_tok);
size_t fold_smem_bytes(const Pool &pool);

// Instantiate BODY (which names the dstate as NN) for each supported dstate.
#define SSM_DISPATCH_N(N_, ...)                               \
    switch (N_) {                                             \
    case 16: { constexpr int NN = 16; __VA_ARGS__; } break;   \
    case 32: { constexpr int NN = 32; __VA_ARGS__; } break;   \
    case 64: { constexpr int NN = 64; __VA_ARGS__; } break;   \
    case 128: { constexpr int NN = 128; __VA_ARGS__; } break; \
    case 256: { constexpr int NN = 256; __VA_ARGS__; } break; \
    default: return cudaErrorInvalidValue;                    \
    }

// ---------------------------------------------------------------- device helpers

// Prefix sums of dt kept as unevaluated pairs hi + lo of fp32 values: each
// addition also carries its rounding error (Knuth's two-sum), so the
// difference of two prefix sums is as accurate as its fp32 result can hold
// (a sum of the dt between two tokens, the exponent of a decay factor)
// without fp64 arithmetic, whose throughput on this GPU is a small fraction
// of fp32's.  No multiplies are involved, so FMA contraction cannot change it.
struct Sum2 {
    float hi, lo;
};

__device__ __forceinline__ Sum2 sum2_add(Sum2 a, Sum2 b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float e = ((a.hi - (s - bb)) + (b.hi - bb)) + (a.lo + b.lo);
    const float hi = s + e;
    return Sum2{hi, e - (hi - s)};
}

__device__ __forceinline__ float sum2_diff(Sum2 a, Sum2 b) { return (a.hi - b.hi) + (a.lo - b.lo); }

// Inclusive prefix sums of dt[0 .. m) into cum[0 .. m) by one warp.
__device__ __forceinline__ void warp_prefix_sum2(const float *dt, Sum2 *cum, int m, int lane) {
    Sum2 carry{0.f, 0.f};
    for (int base = 0; base < m; base += 32) {
        const int s = base + lane;
        Sum2 v{s < m ? dt[s] : 0.f, 0.f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const Sum2 u{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
            if (lane >= o) v = sum2_add(u, v);
        }
        if (s < m) cum[s] = sum2_add(carry, v);
        carry = sum2_add(carry, Sum2{__shfl_sync(0xffffffffu, v.hi, 31), __shfl_sync(0xffffffffu, v.lo, 31)});
    }
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float load_dt(const void *dt, size_t idx, int is_bf16) {
    return is_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(dt)[idx])
                   : reinterpret_cast<const float *>(dt)[idx];
}

// Four consecutive input values starting at element e (e multiple of 4).
__device__ __forceinline__ float4 load4(const float *p, size_t e) {
    return *reinterpret_cast<const float4 *>(p + e);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p, size_t e) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p + e);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ bool finite4(float4 v) {
    return isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w);
}

// The lane's 16 values of a length-N vector (see the layout note above).
template <int N, typename T>
__device__ __forceinline__ void load_lane16(const T *v, int sub, float (&out)[16]) {
    constexpr int LPR = N / 16;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = load4(v, (size_t)4 * (sub + LPR * q));
        out[4 * q + 0] = f.x; out[4 * q + 1] = f.y; out[4 * q + 2] = f.z; out[4 * q + 3] = f.w;
    }
}

template <int LPR>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Current state of (slot, head h).  Copy pools keep a slot's current state
// either in the base array (cur = -1) or in snapshot cur after a commit.
__device__ __forceinline__ float *current_state(float *state, float *snap, const int32_t *cur, int n_slots,
                                                size_t hpn, size_t pn, int slot, int h) {
    const size_t off = (size_t)slot * hpn + (size_t)h * pn;
    if (snap != nullptr) {
        const int c = cur[slot];
        if (c >= 0) return snap + (size_t)c * n_slots * hpn + off;
    }
    return state + off;
}

// Packed two-wide fp32 FMA (one instruction, each lane rounded like fmaf).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(*reinterpret_cast<unsigned long long *>(&d))
        : "l"(*reinterpret_cast<const unsigned long long *>(&a)), "l"(*reinterpret_cast<const unsigned long long *>(&b)),
          "l"(*reinterpret_cast<const unsigned long long *>(&c)));
    return d;
}

__device__ __forceinline__ float4 ld_stream(const float *p) { return __ldcs(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ void st_stream(float *p, float4 v) { __stcs(reinterpret_cast<float4 *>(p), v); }

}  // namespace ssm
