// Host side of libssmstate: the C ABI declared in include/ssm_state.h.
//
// The pool is the stream-owned record of Mamba Streaming State That Survives
// Chunking (Treat Mamba streaming state as a stream-owned record): slots are
// named explicitly by every call and validated here, never picked by shape;
// the chunk sequence of each slot is checked on the host before any work is
// queued, so a rejected call leaves everything as it was.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>

#include "ssm_internal.cuh"

using ssm::Pool;

struct ssm_pool_s {
    Pool p;
    std::vector<uint32_t> stamp;  // duplicate-slot detection
    uint32_t gen = 0;
};

namespace {

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

inline ssm_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SSM_OK;
    if (e == cudaErrorMemoryAllocation) return SSM_ERR_NO_MEMORY;
    return SSM_ERR_CUDA;
}

template <typename T>
cudaError_t alloc(T **ptr, size_t count, size_t &bytes) {
    *ptr = nullptr;
    if (count == 0) return cudaSuccess;
    bytes += count * sizeof(T);
    return cudaMalloc(reinterpret_cast<void **>(ptr), count * sizeof(T));
}

void free_all(Pool &p) {
    cudaFree(p.state);
    cudaFree(p.snap);
    cudaFree(p.log_x);
    cudaFree(p.log_dt);
    cudaFree(p.log_B);
    cudaFree(p.d_position);
    cudaFree(p.d_log_len);
    cudaFree(p.d_cur);
    cudaFree(p.d_slot_flags);
    cudaFree(p.d_flags);
    cudaFree(p.d_stage);
    cudaFree(p.d_cb);
    cudaFree(p.d_wsc);
    cudaFree(p.d_dec);
    cudaFree(p.d_cf);
    cudaFree(p.d_fold_items);
    cudaFree(p.d_fold_count);
    cudaFree(p.d_stage_pos);
    cudaFree(p.d_plain);
    cudaFree(p.d_fv_items);
    cudaFree(p.d_moves);
    cudaFree(p.d_counts);
    Pool::HostPipe &h = p.hpipe;
    cudaFree(h.buf);
    for (cudaEvent_t e : {h.start, h.in_ready[0], h.in_ready[1], h.used[0], h.used[1], h.y_ready[0], h.y_ready[1],
                          h.y_free[0], h.y_free[1]})
        if (e) cudaEventDestroy(e);
    if (h.up) cudaStreamDestroy(h.up);
    if (h.down) cudaStreamDestroy(h.down);
    h = Pool::HostPipe{};
}

int warps_needed(int N, int P) {
    const int rows = (32 / (N / 16)) * ssm::kRowsPerThread;
    return (P + rows - 1) / rows;
}

// Slots: in range, distinct, and (unless allow_released) not released.
ssm_status check_slots(ssm_pool_s *pool, const int32_t *slots, int n, bool allow_released) {
    if (!slots || n < 1) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    if (++pool->gen == 0) {
        std::fill(pool->stamp.begin(), pool->stamp.end(), 0u);
        pool->gen = 1;
    }
    for (int i = 0; i < n; ++i) {
        const int s = slots[i];
        if (s < 0 || s >= p.n_slots) return SSM_ERR_INVALID_ARG;
        if (pool->stamp[s] == pool->gen) return SSM_ERR_INVALID_ARG;
        pool->stamp[s] = pool->gen;
    }
    if (!allow_released)
        for (int i = 0; i < n; ++i)
            if (p.released[slots[i]]) return SSM_ERR_INVALID_STATE;
    return SSM_OK;
}

void fill_step(const Pool &p, ssm::StepArgs &a, const void *x, const void *dt, const void *B, const void *C,
               const float *A, const float *D, void *y, int n_tok) {
    std::memset(&a, 0, offsetof(ssm::StepArgs, slots));
    a.x = x; a.dt = dt; a.B = B; a.C = C; a.A = A; a.D = D; a.y = y;
    a.state = p.state; a.snap = p.snap;
    a.log_x = p.log_x; a.log_dt = p.log_dt; a.log_B = p.log_B;
    a.cb = p.d_cb;
    a.cb_w = p.cb_w;
    a.wsc = p.d_wsc;
    a.dec = p.d_dec;
    a.cf = p.d_cf;
    a.t1pad = p.t1pad;
    a.cf_rows = p.cf_rows;
    a.position = p.d_position; a.log_len = p.d_log_len; a.cur = p.d_cur;
    a.slot_flags = p.d_slot_flags; a.flags = p.d_flags;
    a.H = p.H; a.P = p.P; a.N = p.N; a.G = p.G; a.hpg = p.hpg;
    a.n_slots = p.n_slots; a.t1max = p.t1max; a.wcap = p.wcap;
    a.n_tok = n_tok;
    a.dt_bf16 = p.cfg.dt_dtype == SSM_DTYPE_BF16;
    a.check_log = p.cfg.mode == SSM_MODE_REPLAY;
    a.wwin = p.wwin;
    if (p.fold_in_verify) {
        a.fold_w = p.cfg.window;
        a.stage_pos = p.d_stage_pos;
        a.plain = p.d_plain;
        a.fv_items = p.d_fv_items;
        a.counts = p.d_counts;
    }
}

void fill_commit(const Pool &p, ssm::CommitArgs &c, const float *A) {
    std::memset(&c, 0, offsetof(ssm::CommitArgs, slots));
    c.A = A; c.state = p.state;
    c.log_x = p.log_x; c.log_dt = p.log_dt; c.log_B = p.log_B;
    c.position = p.d_position; c.log_len = p.d_log_len; c.cur = p.d_cur;
    c.slot_flags = p.d_slot_flags; c.flags = p.d_flags;
    c.H = p.H; c.P = p.P; c.N = p.N; c.G = p.G; c.hpg = p.hpg;
    c.n_slots = p.n_slots; c.t1max = p.t1max; c.wcap = p.wcap; c.W = p.cfg.window;
    c.fold_items = p.d_fold_items; c.fold_count = p.d_fold_count;
    c.wwin = p.wwin;
    if (p.fold_in_verify) {
        c.fold_w = p.cfg.window;
        c.stage_pos = p.d_stage_pos;
        c.moves = p.d_moves;
        c.counts = p.d_counts;
    }
}

size_t in_elem(int dtype) { return dtype == SSM_DTYPE_BF16 ? 2 : 4; }

// Launch a per-slot step over batches of at most kMaxSlotsPerLaunch slots,
// advancing the token-major input / output pointers by the slots done.
template <typename Launch>
ssm_status run_step(const Pool &p, ssm::StepArgs &a, const int32_t *slots, int batch, int n_tok, Launch launch,
                    cudaStream_t s) {
    const size_t in_b = in_elem(p.cfg.input_dtype), dt_b = in_elem(p.cfg.dt_dtype);
    const char *x0 = static_cast<const char *>(a.x), *dt0 = static_cast<const char *>(a.dt);
    const char *B0 = static_cast<const char *>(a.B), *C0 = static_cast<const char *>(a.C);
    char *y0 = static_cast<char *>(a.y);
    for (int base = 0; base < batch; base += ssm::kMaxSlotsPerLaunch) {
        const int m = std::min(batch - base, ssm::kMaxSlotsPerLaunch);
        const size_t tok = (size_t)base * n_tok;
        a.x = x0 + tok * p.H * p.P * in_b;
        a.dt = dt0 + tok * p.H * dt_b;
        a.B = B0 + tok * p.G * p.N * in_b;
        a.C = C0 + tok * p.G * p.N * in_b;
        a.y = y0 + tok * p.H * p.P * in_b;
        a.batch = m;
        for (int i = 0; i < m; ++i) a.slots[i] = slots[base + i];
        const cudaError_t e = launch(p, a, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return SSM_OK;
}

}  // namespace

extern "C" {

const char *ssm_status_string(ssm_status s) {
    switch (s) {
    case SSM_OK: return "ok";
    case SSM_ERR_INVALID_ARG: return "invalid argument";
    case SSM_ERR_INVALID_CHUNK: return "invalid_chunk";
    case SSM_ERR_INVALID_STATE: return "invalid_state";
    case SSM_ERR_SEQUENCE: return "chunk sequence out of order";
    case SSM_ERR_DUPLICATE: return "chunk already applied";
    case SSM_ERR_SCHEMA: return "state schema mismatch";
    case SSM_ERR_CUDA: return "CUDA error";
    case SSM_ERR_TIMEOUT: return "device wait timed out";
    case SSM_ERR_NO_MEMORY: return "out of memory";
    }
    return "unknown status";
}

ssm_status ssm_state_init(const ssm_config *cfg, int32_t n_slots, const float *init_state, ssm_stream_t stream,
                          ssm_pool *out) {
    if (!cfg || !out || n_slots < 1) return SSM_ERR_INVALID_ARG;
    const ssm_config c = *cfg;
    const bool n_ok = c.dstate == 16 || c.dstate == 32 || c.dstate == 64 || c.dstate == 128 || c.dstate == 256;
    if (c.nheads < 1 || c.headdim < 1 || c.headdim > 256 || !n_ok || c.ngroups < 1 || c.nheads % c.ngroups)
        return SSM_ERR_INVALID_ARG;
    if ((c.input_dtype != SSM_DTYPE_F32 && c.input_dtype != SSM_DTYPE_BF16) ||
        (c.dt_dtype != SSM_DTYPE_F32 && c.dt_dtype != SSM_DTYPE_BF16))
        return SSM_ERR_INVALID_ARG;
    if (c.mode != SSM_MODE_COPY && c.mode != SSM_MODE_REPLAY) return SSM_ERR_INVALID_ARG;
    if (c.max_tokens < 1 || c.max_tokens > 64) return SSM_ERR_INVALID_ARG;
    if (c.mode == SSM_MODE_REPLAY && (c.window < 1 || c.window > 1024)) return SSM_ERR_INVALID_ARG;
    if (c.fold != SSM_FOLD_AT_COMMIT && c.fold != SSM_FOLD_IN_VERIFY) return SSM_ERR_INVALID_ARG;
    const bool fiv = c.fold == SSM_FOLD_IN_VERIFY;
    if (fiv && (c.mode != SSM_MODE_REPLAY || c.input_dtype != SSM_DTYPE_BF16 || c.headdim != 64 || c.dstate != 128 ||
                (c.nheads / c.ngroups) % 2 != 0 || c.max_tokens > 32 || c.window - 1 + 2 * c.max_tokens > 64))
        return SSM_ERR_INVALID_ARG;
    if (32 * warps_needed(c.dstate, c.headdim) > ssm::kMaxThreads) return SSM_ERR_INVALID_ARG;

    ssm_pool_s *pool = new (std::nothrow) ssm_pool_s();
    if (!pool) return SSM_ERR_NO_MEMORY;
    Pool &p = pool->p;
    p.cfg = c;
    p.n_slots = n_slots;
    p.H = c.nheads; p.P = c.headdim; p.N = c.dstate; p.G = c.ngroups; p.hpg = c.nheads / c.ngroups;
    p.pn = (size_t)p.P * p.N;
    p.hpn = (size_t)p.H * p.pn;
    p.t1max = c.max_tokens;
    p.fold_in_verify = fiv;
    p.wwin = c.mode == SSM_MODE_REPLAY ? c.window - 1 + c.max_tokens : 0;
    // a verify that folds stages its tokens after a log of up to W - 1 + t1max
    p.wcap = p.wwin + (fiv ? c.max_tokens : 0);
    p.cb_w = (p.wwin + 3) / 4 * 4;
    if (c.mode == SSM_MODE_REPLAY && p.wwin <= 32) p.cb_w = 32;  // whole-row float4 reads of the W rows
    p.t1pad = (p.t1max + 3) / 4 * 4;
    p.cf_rows = (p.t1max + 15) / 16 * 16;
    p.in_bytes = in_elem(c.input_dtype);
    if (cudaGetDevice(&p.device) != cudaSuccess) { delete pool; return SSM_ERR_CUDA; }
    if (cudaDeviceGetAttribute(&p.sm_count, cudaDevAttrMultiProcessorCount, p.device) != cudaSuccess || p.sm_count < 1)
        p.sm_count = 1;
    p.cb_rows = std::min(n_slots, ssm::kMaxSlotsPerLaunch);

    if (c.mode == SSM_MODE_REPLAY && !fiv) {  // the kernels a pool that folds in its verify never runs
        int max_smem = 0;
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, p.device);
        if (ssm::replay_smem_bytes(p, c.max_tokens) > (size_t)max_smem ||
            ssm::replay_prep_smem_bytes(p, c.max_tokens) > (size_t)max_smem ||
            ssm::fold_smem_bytes(p) > (size_t)max_smem) {
            delete pool;
            return SSM_ERR_INVALID_ARG;
        }
    }

    cudaError_t e = cudaSuccess;
    size_t &b = p.bytes;
    const size_t ns = (size_t)n_slots;
    if (e == cudaSuccess) e = alloc(&p.state, ns * p.hpn, b);
    if (e == cudaSuccess && c.mode == SSM_MODE_COPY) e = alloc(&p.snap, 2 * (size_t)p.t1max * ns * p.hpn, b);
    if (e == cudaSuccess && c.mode == SSM_MODE_REPLAY) {
        char *lx = nullptr, *lB = nullptr;
        e = alloc(&lx, ns * p.wcap * p.H * p.P * p.in_bytes, b);
        p.log_x = lx;
        if (e == cudaSuccess) e = alloc(&p.log_dt, ns * p.wcap * p.H, b);
        if (e == cudaSuccess) e = alloc(&lB, ns * p.wcap * p.G * p.N * p.in_bytes, b);
        p.log_B = lB;
        if (e == cudaSuccess) e = alloc(&p.d_cb, (size_t)p.cb_rows * p.G * p.t1max * p.cb_w, b);
        if (e == cudaSuccess) e = alloc(&p.d_wsc, (size_t)p.cb_rows * p.H * p.t1max * p.cb_w, b);
        if (e == cudaSuccess) e = alloc(&p.d_dec, (size_t)p.cb_rows * p.H * p.t1pad, b);
        if (e == cudaSuccess) e = alloc(&p.d_cf, (size_t)p.cb_rows * p.G * p.cf_rows * p.N, b);
        if (e == cudaSuccess) e = alloc(&p.d_fold_items, (size_t)ssm::kMaxSlotsPerLaunch, b);
        if (e == cudaSuccess) e = alloc(&p.d_fold_count, 1, b);
    }
    if (e == cudaSuccess && fiv) {
        e = alloc(&p.d_stage_pos, ns, b);
        if (e == cudaSuccess) e = alloc(&p.d_plain, (size_t)ssm::kMaxSlotsPerLaunch, b);
        if (e == cudaSuccess) e = alloc(&p.d_fv_items, (size_t)ssm::kMaxSlotsPerLaunch, b);
        if (e == cudaSuccess) e = alloc(&p.d_moves, (size_t)ssm::kMaxSlotsPerLaunch, b);
        if (e == cudaSuccess) e = alloc(&p.d_counts, 4, b);
    }
    if (e == cudaSuccess) e = alloc(&p.d_position, ns, b);
    if (e == cudaSuccess) e = alloc(&p.d_log_len, ns, b);
    if (e == cudaSuccess) e = alloc(&p.d_cur, ns, b);
    if (e == cudaSuccess) e = alloc(&p.d_slot_flags, ns, b);
    if (e == cudaSuccess) e = alloc(&p.d_flags, 1, b);
    if (e == cudaSuccess) e = alloc(&p.d_stage, p.hpn, b);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (e == cudaSuccess) {
        if (init_state) e = cudaMemcpyAsync(p.state, init_state, ns * p.hpn * sizeof(float), cudaMemcpyDeviceToDevice, s);
        else e = cudaMemsetAsync(p.state, 0, ns * p.hpn * sizeof(float), s);
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(p.d_position, 0, ns * sizeof(int64_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.d_log_len, 0, ns * sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.d_cur, 0xff, ns * sizeof(int32_t), s);  // -1: base state
    if (e == cudaSuccess) e = cudaMemsetAsync(p.d_slot_flags, 0, ns * sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.d_flags, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess && fiv) e = cudaMemsetAsync(p.d_stage_pos, 0, ns * sizeof(int32_t), s);
    if (e == cudaSuccess && fiv) e = cudaMemsetAsync(p.d_counts, 0, 4 * sizeof(int32_t), s);
    if (e == cudaSuccess && c.mode == SSM_MODE_REPLAY) {  // padding rows of the scratch read as zeros
        e = cudaMemsetAsync(p.d_cf, 0, (size_t)p.cb_rows * p.G * p.cf_rows * p.N * sizeof(float), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(p.d_wsc, 0, (size_t)p.cb_rows * p.H * p.t1max * p.cb_w * sizeof(float), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(p.d_dec, 0, (size_t)p.cb_rows * p.H * p.t1pad * sizeof(float), s);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        free_all(p);
        delete pool;
        return cuda_status(e);
    }
    if (c.mode == SSM_MODE_REPLAY) ssm::replay_tma_encode(p);  // else the bulk-copy / plain kernels serve
    if (fiv && (!p.tm_tc_ok || !p.tm_fold_ok || !ssm::fold_verify_fits(p))) {  // the verify's fold needs them
        free_all(p);
        delete pool;
        return SSM_ERR_INVALID_ARG;
    }
    p.next_chunk.assign(ns, 0);
    p.epoch.assign(ns, 0);
    p.released.assign(ns, 0);
    p.pending_ntok.assign(ns, 0);
    pool->stamp.assign(ns, 0);
    *out = pool;
    return SSM_OK;
}

ssm_status ssm_state_destroy(ssm_pool pool) {
    if (!pool) return SSM_ERR_INVALID_ARG;
    DeviceGuard g(pool->p.device);
    cudaDeviceSynchronize();
    free_all(pool->p);
    delete pool;
    return SSM_OK;
}

ssm_status ssm_state_reset(ssm_pool pool, const int32_t *slots, int32_t n, ssm_stream_t stream) {
    if (!pool) return SSM_ERR_INVALID_ARG;
    ssm_status st = check_slots(pool, slots, n, true);
    if (st != SSM_OK) return st;
    DeviceGuard g(pool->p.device);
    Pool &p = pool->p;
    const cudaError_t e = ssm::launch_reset(p, slots, n, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    for (int i = 0; i < n; ++i) {
        const int s = slots[i];
        p.next_chunk[s] = 0;
        p.epoch[s] += 1;
        p.released[s] = 0;
        p.pending_ntok[s] = 0;
    }
    p.last_path = "reset";
    return SSM_OK;
}

ssm_status ssm_state_release(ssm_pool pool, const int32_t *slots, int32_t n) {
    if (!pool) return SSM_ERR_INVALID_ARG;
    ssm_status st = check_slots(pool, slots, n, false);
    if (st != SSM_OK) return st;
    for (int i = 0; i < n; ++i) {
        pool->p.released[slots[i]] = 1;
        pool->p.pending_ntok[slots[i]] = 0;
    }
    return SSM_OK;
}

static ssm_status read_meta(ssm_pool pool, int32_t slot, ssm_slot_meta *meta, cudaStream_t s) {
    Pool &p = pool->p;
    int64_t pos = 0;
    int32_t ll = 0;
    uint32_t fl = 0;
    cudaError_t e = cudaMemcpyAsync(&pos, p.d_position + slot, sizeof(pos), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&ll, p.d_log_len + slot, sizeof(ll), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&fl, p.d_slot_flags + slot, sizeof(fl), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    meta->position = pos;
    meta->next_chunk = p.next_chunk[slot];
    meta->epoch = p.epoch[slot];
    meta->log_len = ll;
    meta->flags = (fl & ssm::kSlotPoisoned ? 1u : 0u) | (p.released[slot] ? 2u : 0u);
    return SSM_OK;
}

ssm_status ssm_slot_info(ssm_pool pool, int32_t slot, ssm_slot_meta *meta, ssm_stream_t stream) {
    if (!pool || !meta || slot < 0 || slot >= pool->p.n_slots) return SSM_ERR_INVALID_ARG;
    DeviceGuard g(pool->p.device);
    return read_meta(pool, slot, meta, reinterpret_cast<cudaStream_t>(stream));
}

ssm_status ssm_state_checkpoint(ssm_pool pool, int32_t slot, const float *A, float *host_state, size_t cap_bytes,
                                ssm_slot_meta *meta, ssm_stream_t stream) {
    if (!pool || !host_state || !meta || slot < 0 || slot >= pool->p.n_slots) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    if (cap_bytes < p.hpn * sizeof(float)) return SSM_ERR_INVALID_ARG;
    if (p.released[slot]) return SSM_ERR_INVALID_STATE;
    DeviceGuard g(p.device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ssm_slot_meta m0;
    ssm_status st = read_meta(pool, slot, &m0, s);
    if (st != SSM_OK) return st;
    if (m0.flags & 1u) return SSM_ERR_INVALID_STATE;  // poisoned: nothing valid to save
    if (p.cfg.mode == SSM_MODE_REPLAY && m0.log_len > 0) {
        if (!A) return SSM_ERR_INVALID_ARG;
        ssm::CommitArgs c;
        fill_commit(p, c, A);
        c.fold_grid = p.H;
        c.flush = 1; c.batch = 1;
        c.slots[0] = slot;
        c.ntok[0] = 1;
        const cudaError_t e = ssm::launch_commit(p, c, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    cudaError_t e = ssm::launch_gather(p, &slot, 1, p.d_stage, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(host_state, p.d_stage, p.hpn * sizeof(float), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    p.last_path = "checkpoint";
    return read_meta(pool, slot, meta, s);
}

ssm_status ssm_state_restore(ssm_pool pool, int32_t slot, const float *host_state, size_t bytes,
                             const ssm_slot_meta *meta, ssm_stream_t stream) {
    if (!pool || !host_state || !meta || slot < 0 || slot >= pool->p.n_slots) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    if (bytes != p.hpn * sizeof(float)) return SSM_ERR_SCHEMA;
    if (meta->position < 0 || meta->next_chunk < 0 || meta->epoch < 0) return SSM_ERR_SCHEMA;
    DeviceGuard g(p.device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t pos = meta->position;
    const int32_t zero = 0, minus1 = -1;
    const uint32_t clear = 0;
    cudaError_t e = cudaMemcpyAsync(p.state + (size_t)slot * p.hpn, host_state, bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p.d_position + slot, &pos, sizeof(pos), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p.d_log_len + slot, &zero, sizeof(zero), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p.d_cur + slot, &minus1, sizeof(minus1), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(p.d_slot_flags + slot, &clear, sizeof(clear), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    p.next_chunk[slot] = meta->next_chunk;
    p.epoch[slot] = meta->epoch;
    p.released[slot] = 0;
    p.pending_ntok[slot] = 0;
    p.last_path = "restore";
    return SSM_OK;
}

ssm_status ssm_state_checkpoint_receipt(ssm_pool pool, int32_t slot, const float *A, const ssm_stream_identity *id,
                                        void *buf, size_t cap, size_t *written, ssm_stream_t stream) {
    if (!pool || !id) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    const size_t need = ssm_receipt_bytes(p.H, p.P, p.N);
    if (written) *written = need;
    if (!buf || cap < need) return SSM_ERR_INVALID_ARG;
    std::vector<float> host(p.hpn);
    ssm_slot_meta meta;
    ssm_status st = ssm_state_checkpoint(pool, slot, A, host.data(), host.size() * sizeof(float), &meta, stream);
    if (st != SSM_OK) return st;
    ssm_receipt r;
    std::memset(&r, 0, sizeof(r));
    r.id = *id;
    r.schema_version = SSM_STATE_SCHEMA_VERSION;
    r.state_dtype = SSM_DTYPE_F32;
    r.input_dtype = p.cfg.input_dtype;
    r.dt_dtype = p.cfg.dt_dtype;
    r.nheads = p.H; r.headdim = p.P; r.dstate = p.N; r.ngroups = p.G;
    r.position = meta.position;
    r.next_chunk = meta.next_chunk;
    return ssm_receipt_encode(&r, host.data(), buf, cap, written);
}

ssm_status ssm_state_restore_receipt(ssm_pool pool, int32_t slot, const void *buf, size_t len,
                                     const ssm_stream_identity *expect, ssm_stream_t stream) {
    if (!pool || !buf || !expect || slot < 0 || slot >= pool->p.n_slots) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    ssm_receipt r;
    const void *payload = nullptr;
    ssm_status st = ssm_receipt_decode(buf, len, &r, &payload);
    if (st != SSM_OK) return st;
    // every semantic field must match: whose state, which layout, precision and shape
    if (r.id.stream_id != expect->stream_id || r.id.model_revision != expect->model_revision ||
        r.id.code_revision != expect->code_revision || r.id.layer != expect->layer)
        return SSM_ERR_SCHEMA;
    if (r.schema_version != SSM_STATE_SCHEMA_VERSION || r.state_dtype != SSM_DTYPE_F32 ||
        r.input_dtype != p.cfg.input_dtype || r.dt_dtype != p.cfg.dt_dtype)
        return SSM_ERR_SCHEMA;
    if (r.nheads != p.H || r.headdim != p.P || r.dstate != p.N || r.ngroups != p.G) return SSM_ERR_SCHEMA;
    if (r.position < 0 || r.next_chunk < 0) return SSM_ERR_SCHEMA;
    std::vector<float> host(p.hpn);
    std::memcpy(host.data(), payload, p.hpn * sizeof(float));  // the blob holds little-endian fp32
    ssm_slot_meta meta;
    std::memset(&meta, 0, sizeof(meta));
    meta.position = r.position;
    meta.next_chunk = r.next_chunk;
    meta.epoch = p.epoch[slot] + 1;  // a new occupant of the slot
    st = ssm_state_restore(pool, slot, host.data(), host.size() * sizeof(float), &meta, stream);
    if (st == SSM_OK) p.last_path = "restore_receipt";
    return st;
}

ssm_status ssm_state_gather(ssm_pool pool, int32_t n, const int32_t *slots, float *dst, ssm_stream_t stream) {
    if (!pool || !dst) return SSM_ERR_INVALID_ARG;
    ssm_status st = check_slots(pool, slots, n, true);
    if (st != SSM_OK) return st;
    DeviceGuard g(pool->p.device);
    return cuda_status(ssm::launch_gather(pool->p, slots, n, dst, reinterpret_cast<cudaStream_t>(stream)));
}

ssm_status ssm_scan_chunk(ssm_pool pool, int32_t n_seq, const int32_t *cu_seqlens, const int32_t *slots,
                          const int64_t *chunk_seq, const void *x, const void *dt, const void *B, const void *C,
                          const float *A, const float *D, void *y, ssm_stream_t stream) {
    if (!pool || !cu_seqlens || !chunk_seq || n_seq < 1) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    if (cu_seqlens[0] != 0) return SSM_ERR_INVALID_ARG;
    for (int i = 0; i < n_seq; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return SSM_ERR_INVALID_ARG;
    const int64_t total = cu_seqlens[n_seq];
    if (total > 0 && (!x || !dt || !B || !C || !A || !D || !y)) return SSM_ERR_INVALID_ARG;
    ssm_status st = check_slots(pool, slots, n_seq, false);
    if (st != SSM_OK) return st;
    for (int i = 0; i < n_seq; ++i) {  // declared mismatch, before anything advances
        const int64_t want = p.next_chunk[slots[i]];
        if (chunk_seq[i] < want) return SSM_ERR_DUPLICATE;
        if (chunk_seq[i] > want) return SSM_ERR_SEQUENCE;
    }
    DeviceGuard g(p.device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (total > 0) {
        ssm::ScanArgs a;
        std::memset(&a, 0, offsetof(ssm::ScanArgs, cu));
        a.x = x; a.dt = dt; a.B = B; a.C = C; a.A = A; a.D = D; a.y = y;
        a.state = p.state; a.snap = p.snap; a.cur = p.d_cur; a.n_slots = p.n_slots;
        a.position = p.d_position; a.log_len = p.d_log_len;
        a.slot_flags = p.d_slot_flags; a.flags = p.d_flags;
        a.H = p.H; a.P = p.P; a.N = p.N; a.G = p.G; a.hpg = p.hpg;
        a.dt_bf16 = p.cfg.dt_dtype == SSM_DTYPE_BF16;
        a.check_log = p.cfg.mode == SSM_MODE_REPLAY;
        for (int base = 0; base < n_seq; base += ssm::kMaxSeqPerLaunch) {
            const int m = std::min(n_seq - base, ssm::kMaxSeqPerLaunch);
            a.n_seq = m;
            for (int i = 0; i <= m; ++i) a.cu[i] = cu_seqlens[base + i];
            for (int i = 0; i < m; ++i) a.slots[i] = slots[base + i];
            // the tensor-core scan moves x, B, C and y in 16-byte pieces
            const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(B) |
                                   reinterpret_cast<uintptr_t>(C) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
            const char *path = "scan_seq";
            bool ssd = aligned && ssm::scan_ssd_supported(p);
            cudaError_t e = ssd ? ssm::launch_scan_ssd(p, a, s, &path) : cudaErrorNotSupported;
            if (e == cudaErrorNotSupported) {  // no tensor maps for these buffers: the sequential scan
                path = "scan_seq";
                e = ssm::launch_scan_seq(p, a, s);
            }
            if (e != cudaSuccess) return cuda_status(e);
            p.last_path = path;
        }
    }
    for (int i = 0; i < n_seq; ++i) {
        p.next_chunk[slots[i]] += 1;
        p.pending_ntok[slots[i]] = 0;
    }
    return SSM_OK;
}

ssm_status ssm_decode_step(ssm_pool pool, int32_t batch, const int32_t *slots, const void *x, const void *dt,
                           const void *B, const void *C, const float *A, const float *D, void *y,
                           ssm_stream_t stream) {
    if (!pool || !x || !dt || !B || !C || !A || !D || !y) return SSM_ERR_INVALID_ARG;
    ssm_status st = check_slots(pool, slots, batch, false);
    if (st != SSM_OK) return st;
    Pool &p = pool->p;
    DeviceGuard g(p.device);
    ssm::StepArgs a;
    fill_step(p, a, x, dt, B, C, A, D, y, 1);
    st = run_step(p, a, slots, batch, 1, ssm::launch_decode, reinterpret_cast<cudaStream_t>(stream));
    if (st != SSM_OK) return st;
    for (int i = 0; i < batch; ++i) p.pending_ntok[slots[i]] = 0;
    p.last_path = "decode";
    return SSM_OK;
}

// The host pipe's streams and events, and staging sets of at least set_bytes
// (re-allocated once the previous sets are idle).
static cudaError_t host_pipe_ready(Pool &p, size_t set_bytes) {
    Pool::HostPipe &h = p.hpipe;
    cudaError_t e = cudaSuccess;
    if (!h.up) {
        e = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking);
        cudaEvent_t *evs[] = {&h.start, &h.in_ready[0], &h.in_ready[1], &h.used[0], &h.used[1],
                              &h.y_ready[0], &h.y_ready[1], &h.y_free[0], &h.y_free[1]};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
    }
    if (set_bytes <= h.set_cap) return cudaSuccess;
    if (h.buf) {  // queued copies and decodes of earlier calls may still touch the old sets
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            e = cudaEventSynchronize(h.used[b]);
            if (e == cudaSuccess) e = cudaEventSynchronize(h.y_free[b]);
        }
        if (e == cudaSuccess) e = cudaStreamSynchronize(h.up);
        if (e != cudaSuccess) return e;
        cudaFree(h.buf);
        p.bytes -= 2 * h.set_cap;
        h.buf = nullptr;
        h.set_cap = 0;
    }
    const size_t cap = (set_bytes + 255) / 256 * 256;
    e = cudaMalloc(reinterpret_cast<void **>(&h.buf), 2 * cap);
    if (e != cudaSuccess) {
        h.buf = nullptr;
        return e;
    }
    p.bytes += 2 * cap;
    h.set_cap = cap;
    return cudaSuccess;
}

static bool page_locked(const void *ptr) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

ssm_status ssm_decode_steps_host(ssm_pool pool, int32_t batch, const int32_t *slots, int32_t n_steps,
                                 const void *x, const void *dt, const void *B, const void *C, const float *A,
                                 const float *D, void *y, ssm_stream_t stream) {
    if (!pool || !x || !dt || !B || !C || !A || !D || !y || n_steps < 1) return SSM_ERR_INVALID_ARG;
    ssm_status st = check_slots(pool, slots, batch, false);
    if (st != SSM_OK) return st;
    Pool &p = pool->p;
    DeviceGuard g(p.device);
    for (const void *ptr : {x, dt, B, C, static_cast<const void *>(y)})
        if (!page_locked(ptr)) return SSM_ERR_INVALID_ARG;
    const size_t in_b = in_elem(p.cfg.input_dtype), dt_b = in_elem(p.cfg.dt_dtype);
    // one step's bytes of each array; each starts on a 256-byte boundary in a staging set
    const size_t nb[5] = {(size_t)batch * p.H * p.P * in_b, (size_t)batch * p.H * dt_b,
                          (size_t)batch * p.G * p.N * in_b, (size_t)batch * p.G * p.N * in_b,
                          (size_t)batch * p.H * p.P * in_b};
    size_t off[5], set_bytes = 0;
    for (int i = 0; i < 5; ++i) {
        off[i] = set_bytes;
        set_bytes += (nb[i] + 255) / 256 * 256;
    }
    cudaError_t e = host_pipe_ready(p, set_bytes);
    if (e != cudaSuccess) return cuda_status(e);
    Pool::HostPipe &h = p.hpipe;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const char *src[4] = {static_cast<const char *>(x), static_cast<const char *>(dt),
                          static_cast<const char *>(B), static_cast<const char *>(C)};
    char *dst = static_cast<char *>(y);
    e = cudaEventRecord(h.start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h.up, h.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h.down, h.start, 0);
    int b = 0;
    for (int t = 0; t < n_steps && e == cudaSuccess; ++t) {
        b = t & 1;
        char *set = h.buf + b * h.set_cap;
        // inputs of step t into set b, once the decode that last read it is done
        e = cudaStreamWaitEvent(h.up, h.used[b], 0);
        for (int i = 0; i < 4 && e == cudaSuccess; ++i)
            e = cudaMemcpyAsync(set + off[i], src[i] + t * nb[i], nb[i], cudaMemcpyHostToDevice, h.up);
        if (e == cudaSuccess) e = cudaEventRecord(h.in_ready[b], h.up);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h.in_ready[b], 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h.y_free[b], 0);  // set b's output read back
        if (e != cudaSuccess) break;
        ssm::StepArgs a;
        fill_step(p, a, set + off[0], set + off[1], set + off[2], set + off[3], A, D, set + off[4], 1);
        st = run_step(p, a, slots, batch, 1, ssm::launch_decode, s);
        if (st != SSM_OK) return st;
        e = cudaEventRecord(h.used[b], s);
        if (e == cudaSuccess) e = cudaEventRecord(h.y_ready[b], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h.down, h.y_ready[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dst + t * nb[4], set + off[4], nb[4], cudaMemcpyDeviceToHost, h.down);
        if (e == cudaSuccess) e = cudaEventRecord(h.y_free[b], h.down);
    }
    // the last output copy ends after every earlier one (one stream); every input copy was waited on
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, h.y_free[b], 0);
    if (e != cudaSuccess) return cuda_status(e);
    for (int i = 0; i < batch; ++i) p.pending_ntok[slots[i]] = 0;
    p.last_path = "decode";
    return SSM_OK;
}

static ssm_status verify_common(ssm_pool pool, int32_t batch, int32_t n_tok, const int32_t *slots, const void *x,
                                const void *dt, const void *B, const void *C, const float *A, const float *D,
                                void *y, ssm_stream_t stream, int mode) {
    if (!pool || !x || !dt || !B || !C || !A || !D || !y) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    if (p.cfg.mode != mode) return SSM_ERR_INVALID_ARG;
    if (n_tok < 1 || n_tok > p.t1max) return SSM_ERR_INVALID_ARG;
    if (p.fold_in_verify && (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(B) % 16 ||
                             reinterpret_cast<uintptr_t>(C) % 16))
        return SSM_ERR_INVALID_ARG;  // the tensor-core path, the only one that folds, moves rows in 16 bytes
    ssm_status st = check_slots(pool, slots, batch, false);
    if (st != SSM_OK) return st;
    DeviceGuard g(p.device);
    ssm::StepArgs a;
    fill_step(p, a, x, dt, B, C, A, D, y, n_tok);
    a.test_stall = p.test_stall;
    p.test_stall = 0;
    const char *path = mode == SSM_MODE_COPY ? "verify_copy" : "verify_replay";
    auto replay = [&path](const Pool &pl, const ssm::StepArgs &sa, cudaStream_t s) {
        return ssm::launch_verify_replay(pl, sa, s, &path);
    };
    if (mode == SSM_MODE_COPY)
        st = run_step(p, a, slots, batch, n_tok, ssm::launch_verify_copy, reinterpret_cast<cudaStream_t>(stream));
    else
        st = run_step(p, a, slots, batch, n_tok, replay, reinterpret_cast<cudaStream_t>(stream));
    if (st != SSM_OK) return st;
    for (int i = 0; i < batch; ++i) p.pending_ntok[slots[i]] = n_tok;
    p.last_path = path;
    return SSM_OK;
}

ssm_status ssm_verify_copy(ssm_pool pool, int32_t batch, int32_t n_tok, const int32_t *slots, const void *x,
                           const void *dt, const void *B, const void *C, const float *A, const float *D, void *y,
                           ssm_stream_t stream) {
    return verify_common(pool, batch, n_tok, slots, x, dt, B, C, A, D, y, stream, SSM_MODE_COPY);
}

ssm_status ssm_verify_replay(ssm_pool pool, int32_t batch, int32_t n_tok, const int32_t *slots, const void *x,
                             const void *dt, const void *B, const void *C, const float *A, const float *D, void *y,
                             ssm_stream_t stream) {
    return verify_common(pool, batch, n_tok, slots, x, dt, B, C, A, D, y, stream, SSM_MODE_REPLAY);
}

ssm_status ssm_state_commit(ssm_pool pool, int32_t batch, const int32_t *slots, const int32_t *accept,
                            int32_t force_fold, const float *A, ssm_stream_t stream) {
    if (!pool || !accept) return SSM_ERR_INVALID_ARG;
    Pool &p = pool->p;
    if (p.cfg.mode == SSM_MODE_REPLAY && !A) return SSM_ERR_INVALID_ARG;
    ssm_status st = check_slots(pool, slots, batch, false);
    if (st != SSM_OK) return st;
    for (int i = 0; i < batch; ++i)
        if (p.pending_ntok[slots[i]] < 1) return SSM_ERR_INVALID_STATE;
    DeviceGuard g(p.device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ssm::CommitArgs c;
    fill_commit(p, c, A);
    c.force_fold = force_fold ? 1 : 0;
    const char *path = "commit_copy";
    for (int base = 0; base < batch; base += ssm::kMaxSlotsPerLaunch) {
        const int m = std::min(batch - base, ssm::kMaxSlotsPerLaunch);
        c.accept = accept + base;
        c.batch = m;
        c.fold_grid = std::min(m * p.H, 2 * p.sm_count);
        for (int i = 0; i < m; ++i) {
            c.slots[i] = slots[base + i];
            c.ntok[i] = p.pending_ntok[slots[base + i]];
        }
        const cudaError_t e = ssm::launch_commit(p, c, s, &path);
        if (e != cudaSuccess) return cuda_status(e);
    }
    for (int i = 0; i < batch; ++i) p.pending_ntok[slots[i]] = 0;
    p.last_path = path;
    return SSM_OK;
}

ssm_status ssm_pool_status(ssm_pool pool, uint32_t *flags_out, int32_t clear, ssm_stream_t stream) {
    if (!pool || !flags_out) return SSM_ERR_INVALID_ARG;
    DeviceGuard g(pool->p.device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t f = 0;
    cudaError_t e = cudaMemcpyAsync(&f, pool->p.d_flags, sizeof(f), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(pool->p.d_flags, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    *flags_out = f;
    return SSM_OK;
}

const char *ssm_last_path(ssm_pool pool) { return pool ? pool->p.last_path : ssm::static_last_path(); }

size_t ssm_pool_bytes(ssm_pool pool) { return pool ? pool->p.bytes : 0; }

ssm_status ssm_debug_stall_next_verify(ssm_pool pool) {
    if (!pool) return SSM_ERR_INVALID_ARG;
    pool->p.test_stall = 1;
    return SSM_OK;
}

}  // extern "C"
