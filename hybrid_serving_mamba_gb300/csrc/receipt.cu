// Checkpoint receipt and state blob (Mamba Streaming State That Survives
// Chunking, Make reset, checkpoint, and cancellation observable: a receipt
// names the stream, model and code revision, state schema, dtype, layer and
// state dimensions, absolute position, chunk sequence and a checksum, and an
// incompatible resume is refused; the SSM.PREFIX state-store page fixes the
// array blob: uint32 version 1, uint32 number of arrays, then per array its
// rank, shape, dtype code and raw values).  Host code only: nothing here
// touches the device, so the format can be exercised without a GPU.
//
// The checksum is FNV-1a 64 over the blob bytes: offset basis
// 14695981039346656037, and for each byte h = (h xor byte) * 1099511628211
// mod 2^64 (Fowler, Noll and Vo's published definition).
#include <cstring>

#include "ssm_internal.cuh"

namespace {

constexpr char kMagic[4] = {'S', 'S', 'M', 'R'};
constexpr uint32_t kFormat = 1;
constexpr uint32_t kBlobVersion = 1;
constexpr uint32_t kDtypeF32Code = 0;  // the blob's dtype codes: 0 fp32, 1 fp16, 2 bf16
// magic, format, 3 x uint64 identity, layer, schema, 7 x int32, 2 x int64, blob bytes, checksum
constexpr size_t kHeader = 4 + 4 + 24 + 4 + 4 + 7 * 4 + 16 + 8 + 8;
constexpr size_t kBlobHeader = 4 * 7;  // version, n_arrays, ndim, shape[3], dtype code

uint64_t fnv1a64(const unsigned char *p, size_t n) {
    uint64_t h = 14695981039346656037ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 1099511628211ull;
    }
    return h;
}

// Little-endian writers and readers, one byte at a time (the host's own order does not matter).
struct Out {
    unsigned char *p;
    void u32(uint32_t v) {
        for (int i = 0; i < 4; ++i) *p++ = (unsigned char)(v >> (8 * i));
    }
    void u64(uint64_t v) {
        for (int i = 0; i < 8; ++i) *p++ = (unsigned char)(v >> (8 * i));
    }
    void i32(int32_t v) { u32((uint32_t)v); }
    void i64(int64_t v) { u64((uint64_t)v); }
};

struct In {
    const unsigned char *p;
    uint32_t u32() {
        uint32_t v = 0;
        for (int i = 0; i < 4; ++i) v |= (uint32_t)*p++ << (8 * i);
        return v;
    }
    uint64_t u64() {
        uint64_t v = 0;
        for (int i = 0; i < 8; ++i) v |= (uint64_t)*p++ << (8 * i);
        return v;
    }
    int32_t i32() { return (int32_t)u32(); }
    int64_t i64() { return (int64_t)u64(); }
};

bool dims_ok(int32_t H, int32_t P, int32_t N) { return H > 0 && P > 0 && N > 0; }

size_t blob_bytes(int32_t H, int32_t P, int32_t N) { return kBlobHeader + (size_t)H * P * N * sizeof(float); }

}  // namespace

extern "C" {

size_t ssm_receipt_bytes(int32_t nheads, int32_t headdim, int32_t dstate) {
    if (!dims_ok(nheads, headdim, dstate)) return 0;
    return kHeader + blob_bytes(nheads, headdim, dstate);
}

ssm_status ssm_receipt_encode(ssm_receipt *r, const float *state, void *buf, size_t cap, size_t *written) {
    if (!r || !state || !dims_ok(r->nheads, r->headdim, r->dstate)) return SSM_ERR_INVALID_ARG;
    const size_t need = ssm_receipt_bytes(r->nheads, r->headdim, r->dstate);
    if (written) *written = need;
    if (!buf || cap < need) return SSM_ERR_INVALID_ARG;
    unsigned char *base = static_cast<unsigned char *>(buf);
    // the blob first, so that its checksum can go into the receipt
    unsigned char *blob = base + kHeader;
    Out b{blob};
    b.u32(kBlobVersion);
    b.u32(1);  // one array: the ssm state
    b.u32(3);
    b.u32((uint32_t)r->nheads);
    b.u32((uint32_t)r->headdim);
    b.u32((uint32_t)r->dstate);
    b.u32(kDtypeF32Code);
    const size_t n = (size_t)r->nheads * r->headdim * r->dstate;
    for (size_t i = 0; i < n; ++i) {
        uint32_t w;
        std::memcpy(&w, state + i, 4);
        b.u32(w);
    }
    const size_t bb = blob_bytes(r->nheads, r->headdim, r->dstate);
    r->checksum = fnv1a64(blob, bb);
    std::memcpy(base, kMagic, 4);
    Out o{base + 4};
    o.u32(kFormat);
    o.u64(r->id.stream_id);
    o.u64(r->id.model_revision);
    o.u64(r->id.code_revision);
    o.i32(r->id.layer);
    o.u32(r->schema_version);
    o.i32(r->state_dtype);
    o.i32(r->input_dtype);
    o.i32(r->dt_dtype);
    o.i32(r->nheads);
    o.i32(r->headdim);
    o.i32(r->dstate);
    o.i32(r->ngroups);
    o.i64(r->position);
    o.i64(r->next_chunk);
    o.u64((uint64_t)bb);
    o.u64(r->checksum);
    return SSM_OK;
}

ssm_status ssm_receipt_decode(const void *buf, size_t len, ssm_receipt *r, const void **state) {
    if (!buf || !r) return SSM_ERR_INVALID_ARG;
    if (len < kHeader + kBlobHeader) return SSM_ERR_SCHEMA;
    const unsigned char *base = static_cast<const unsigned char *>(buf);
    if (std::memcmp(base, kMagic, 4) != 0) return SSM_ERR_SCHEMA;
    In in{base + 4};
    if (in.u32() != kFormat) return SSM_ERR_SCHEMA;
    ssm_receipt q;
    std::memset(&q, 0, sizeof(q));
    q.id.stream_id = in.u64();
    q.id.model_revision = in.u64();
    q.id.code_revision = in.u64();
    q.id.layer = in.i32();
    q.schema_version = in.u32();
    q.state_dtype = in.i32();
    q.input_dtype = in.i32();
    q.dt_dtype = in.i32();
    q.nheads = in.i32();
    q.headdim = in.i32();
    q.dstate = in.i32();
    q.ngroups = in.i32();
    q.position = in.i64();
    q.next_chunk = in.i64();
    const uint64_t bb = in.u64();
    q.checksum = in.u64();
    if (!dims_ok(q.nheads, q.headdim, q.dstate) || q.ngroups <= 0) return SSM_ERR_SCHEMA;
    if (bb != blob_bytes(q.nheads, q.headdim, q.dstate) || len != kHeader + bb) return SSM_ERR_SCHEMA;
    const unsigned char *blob = base + kHeader;
    if (fnv1a64(blob, bb) != q.checksum) return SSM_ERR_SCHEMA;
    In b{blob};
    if (b.u32() != kBlobVersion || b.u32() != 1 || b.u32() != 3) return SSM_ERR_SCHEMA;
    if (b.u32() != (uint32_t)q.nheads || b.u32() != (uint32_t)q.headdim || b.u32() != (uint32_t)q.dstate)
        return SSM_ERR_SCHEMA;
    if (b.u32() != kDtypeF32Code || q.state_dtype != SSM_DTYPE_F32) return SSM_ERR_SCHEMA;
    *r = q;
    if (state) *state = blob + kBlobHeader;
    return SSM_OK;
}

}  // extern "C"
