// ssu_api.cpp -- the C ABI of libssu (include/ssu.h): argument checks, error
// messages and kernel selection.  Nothing here touches device memory; each
// update call is exactly one kernel launch on the caller's stream.
#include "ssu.h"

#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "ssu_internal.h"
#include "ssu_ssd_params.h"
#include "ssu_verify.h"

namespace {

thread_local char g_err[512] = "";

ssu_status fail(ssu_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

ssu_status ok() { return SSU_OK; }

bool valid_dtype(int32_t d) { return d == SSU_F32 || d == SSU_F16 || d == SSU_BF16; }
bool valid_itype(int32_t t) { return t == SSU_I32 || t == SSU_I64; }

// dstate -> lanes per state row (16 elements per lane), or 0 if unsupported.
int lanes_for(int64_t dstate) {
    switch (dstate) {
    case 16: return 1;
    case 32: return 2;
    case 64: return 4;
    case 128: return 8;
    case 256: return 16;
    }
    return 0;
}

const char *unsupported_name(uint32_t bits) {
    if (bits & SSU_UNSUP_RAND_SEED) return "rand_seed (stochastic rounding is not implemented)";
    if (bits & SSU_UNSUP_STATE_SCALE) return "state_scale";
    if (bits & SSU_UNSUP_INTERMEDIATE) return "intermediate_states_buffer / indices / scales";
    if (bits & SSU_UNSUP_CACHE_STEPS) return "cache_steps != 0";
    if (bits & SSU_UNSUP_ALGORITHM) return "algorithm / backend other than 'auto'";
    return "an unknown argument";
}

ssu_status check_shape(int32_t state_dtype, int32_t io_dtype, int32_t dt_dtype, int64_t heads,
                       int64_t dim, int64_t dstate, int64_t groups, int *lanes) {
    if (!valid_dtype(state_dtype)) return fail(SSU_ERR_INVALID, "state_dtype %d is not an ssu_dtype", state_dtype);
    if (!valid_dtype(io_dtype)) return fail(SSU_ERR_INVALID, "io_dtype %d is not an ssu_dtype", io_dtype);
    if (!valid_dtype(dt_dtype)) return fail(SSU_ERR_INVALID, "dt_dtype %d is not an ssu_dtype", dt_dtype);
    if (heads <= 0 || dim <= 0 || dstate <= 0 || groups <= 0)
        return fail(SSU_ERR_INVALID, "heads, dim, dstate and groups must be positive (got %lld, %lld, %lld, %lld)",
                    (long long)heads, (long long)dim, (long long)dstate, (long long)groups);
    if (heads % groups != 0)
        return fail(SSU_ERR_INVALID, "heads (%lld) must be divisible by groups (%lld)", (long long)heads,
                    (long long)groups);
    if (heads > (1 << 30) || dim > (1 << 30))
        return fail(SSU_ERR_INVALID, "heads and dim must be below 2^30");
    *lanes = lanes_for(dstate);
    if (*lanes == 0)
        return fail(SSU_ERR_UNSUPPORTED, "dstate %lld is not supported (16, 32, 64, 128 or 256)", (long long)dstate);
    return SSU_OK;
}

ssu_status check_strides(const char *name, const int64_t *s) {
    for (int i = 0; i < 3; ++i)
        if (s[i] < 0) return fail(SSU_ERR_INVALID, "%s_stride[%d] is negative", name, i);
    return SSU_OK;
}

ssu_status check_table(const char *name, const ssu_slot_table *t, ssu::SlotTab *out) {
    std::memset(out, 0, sizeof *out);
    if (t == nullptr || t->entries == nullptr) return SSU_OK;
    if (!valid_itype(t->type)) return fail(SSU_ERR_INVALID, "%s table: type %d is not an ssu_itype", name, t->type);
    if (t->mode != SSU_SLOTS_STRIDED && t->mode != SSU_SLOTS_PER_ROW)
        return fail(SSU_ERR_INVALID, "%s table: mode %d is not an ssu_slot_mode", name, t->mode);
    if (t->extent < 0) return fail(SSU_ERR_INVALID, "%s table: negative extent", name);
    if (t->s0 < 0 || t->s1 < 0) return fail(SSU_ERR_INVALID, "%s table: negative stride", name);
    out->entries = t->entries;
    out->s0 = t->s0;
    out->s1 = t->s1;
    out->extent = t->extent;
    out->is_i64 = t->type == SSU_I64;
    out->per_row = t->mode == SSU_SLOTS_PER_ROW;
    return SSU_OK;
}

// Shared checks; fills everything in `kp` except the packed layout.
ssu_status prepare(const ssu_args *a, int64_t rows, const ssu_slot_table *read, const ssu_slot_table *dst,
                   ssu::KParams *kp, int *lanes) {
    if (a == nullptr) return fail(SSU_ERR_INVALID, "args is NULL");
    if (a->unsupported != 0)
        return fail(SSU_ERR_UNSUPPORTED, "not implemented: %s", unsupported_name(a->unsupported));
    if (a->reserved0 != 0) return fail(SSU_ERR_INVALID, "reserved0 must be 0");
    ssu_status st = check_shape(a->state_dtype, a->io_dtype, a->dt_dtype, a->heads, a->dim, a->dstate,
                                a->groups, lanes);
    if (st != SSU_OK) return st;
    if (a->slots <= 0) return fail(SSU_ERR_INVALID, "slots must be positive");
    if (!a->state || !a->A) return fail(SSU_ERR_INVALID, "state and A must not be NULL");
    if (rows > 0 && (!a->x || !a->dt || !a->B || !a->C || !a->y))
        return fail(SSU_ERR_INVALID, "x, dt, B, C and y must not be NULL");
    if (reinterpret_cast<uintptr_t>(a->state) % 16 != 0)
        return fail(SSU_ERR_INVALID, "state must be 16-byte aligned");

    if (rows > 0 && (a->y == a->x || a->y == a->z || a->y == a->dt || a->y == a->B || a->y == a->C ||
                     a->y == a->state))
        return fail(SSU_ERR_INVALID, "y must not alias an input");
    if ((st = check_strides("x", a->x_stride)) || (st = check_strides("dt", a->dt_stride)) ||
        (st = check_strides("B", a->B_stride)) || (st = check_strides("C", a->C_stride)) ||
        (st = check_strides("z", a->z_stride)) || (st = check_strides("y", a->y_stride)))
        return st;
    std::memset(kp, 0, sizeof *kp);
    if ((st = check_table("read", read, &kp->rd)) || (st = check_table("destination", dst, &kp->wr)))
        return st;
    kp->slots = a->slots;
    kp->H = static_cast<int32_t>(a->heads);
    kp->P = static_cast<int32_t>(a->dim);
    kp->N = static_cast<int32_t>(a->dstate);
    kp->G = static_cast<int32_t>(a->groups);
    kp->heads_per_group = static_cast<int32_t>(a->heads / a->groups);
    kp->ptiles = static_cast<int32_t>((a->dim + ssu::kTileRows - 1) / ssu::kTileRows);
    kp->io_dtype = a->io_dtype;
    kp->dt_dtype = a->dt_dtype;
    kp->softplus = a->dt_softplus != 0;
    kp->disable = a->disable_state_update != 0;
    kp->pad = a->pad_slot_id;
    kp->state = a->state;
    kp->x = a->x;
    kp->dt = a->dt;
    kp->B = a->B;
    kp->C = a->C;
    kp->z = a->z;
    kp->A = a->A;
    kp->D = a->D;
    kp->dt_bias = a->dt_bias;
    kp->y = a->y;
    for (int i = 0; i < 3; ++i) {
        kp->xs[i] = a->x_stride[i];
        kp->dts[i] = a->dt_stride[i];
        kp->Bs[i] = a->B_stride[i];
        kp->Cs[i] = a->C_stride[i];
        kp->zs[i] = a->z_stride[i];
        kp->ys[i] = a->y_stride[i];
    }
    kp->status = a->d_status;
    kp->wait_cycles = ssu::kDefaultWaitCycles;
    kp->withhold_unit = -1;
    return SSU_OK;
}

bool aligned16(const void *q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; }

// Which small operands the packed kernel can stage with bulk copies: every
// row it copies (B, C: dstate values of one row and group; x, z, dt: up to 64
// dim rows of one row and head) starts on a 16-byte boundary and is a
// multiple of 16 bytes long.
int32_t packed_bulk_ops(const ssu_args *a) {
    const int64_t io = a->io_dtype == SSU_F32 ? 4 : 2, dts = a->dt_dtype == SSU_F32 ? 4 : 2;
    auto rows_ok = [](const void *base, const int64_t *st, int64_t sz, int64_t count) {
        return base != nullptr && aligned16(base) && st[2] == 1 && (st[0] * sz) % 16 == 0 && (st[1] * sz) % 16 == 0 &&
               (count * sz) % 16 == 0;
    };
    int32_t ops = 0;
    if (rows_ok(a->B, a->B_stride, io, a->dstate) && rows_ok(a->C, a->C_stride, io, a->dstate)) ops |= ssu::kBulkBC;
    if (rows_ok(a->x, a->x_stride, io, a->dim) && (a->z == nullptr || rows_ok(a->z, a->z_stride, io, a->dim)))
        ops |= ssu::kBulkXZ;
    if (rows_ok(a->dt, a->dt_stride, dts, a->dim)) ops |= ssu::kBulkDT;
    return ops;
}

// The kernels launch on the current device: a state pool that lives on
// another device would be addressed from the wrong one.  Checked right before
// a launch, after every host check.
ssu_status check_device(const void *state) {
    int dev = -1;
    cudaPointerAttributes pa;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(SSU_ERR_CUDA, "no current CUDA device");
    if (cudaPointerGetAttributes(&pa, state) != cudaSuccess) {
        cudaGetLastError();
        return fail(SSU_ERR_INVALID, "the state pointer is not one the CUDA runtime knows");
    }
    if (pa.type == cudaMemoryTypeDevice && pa.device != dev)
        return fail(SSU_ERR_INVALID, "the state is on device %d but device %d is current", pa.device, dev);
    return SSU_OK;
}

ssu_status launched(cudaError_t e) {
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return ok();
}

constexpr int64_t kMaxGrid = 0x7fffffffLL;

}  // namespace

extern "C" {

ssu_status ssu_update_onetoken(const ssu_args *args, int64_t batch, const ssu_slot_table *read,
                               const ssu_slot_table *dst, void *stream) {
    ssu::KParams kp;
    int lanes = 0;
    if (batch < 0) return fail(SSU_ERR_INVALID, "batch is negative");
    ssu_status st = prepare(args, batch, read, dst, &kp, &lanes);
    if (st != SSU_OK) return st;
    if (batch == 0) return ok();
    if (batch * kp.H * kp.ptiles > kMaxGrid) return fail(SSU_ERR_INVALID, "batch * heads * dim tiles exceeds 2^31-1");
    kp.nseq = batch;
    kp.rows = batch;
    if ((st = check_device(args->state)) != SSU_OK) return st;
    return launched(ssu::launch_onetoken(args->state_dtype, lanes, kp, batch,
                                         static_cast<cudaStream_t>(stream)));
}

ssu_status ssu_selftest_timeout(const ssu_args *args, int64_t batch, const ssu_slot_table *read,
                                const ssu_slot_table *dst, int64_t withhold_unit, int64_t wait_cycles,
                                void *stream) {
    ssu::KParams kp;
    int lanes = 0;
    if (batch <= 0) return fail(SSU_ERR_INVALID, "batch must be positive");
    ssu_status st = prepare(args, batch, read, dst, &kp, &lanes);
    if (st != SSU_OK) return st;
    if (batch * kp.H * kp.ptiles > kMaxGrid) return fail(SSU_ERR_INVALID, "batch * heads * dim tiles exceeds 2^31-1");
    if (withhold_unit < 0 || withhold_unit >= batch * kp.H * kp.ptiles)
        return fail(SSU_ERR_INVALID, "withhold_unit must name a unit of the call");
    if (wait_cycles < 1000 || wait_cycles > ssu::kDefaultWaitCycles)
        return fail(SSU_ERR_INVALID, "wait_cycles must be in [1000, %lld]", (long long)ssu::kDefaultWaitCycles);
    kp.nseq = batch;
    kp.rows = batch;
    kp.withhold_unit = withhold_unit;
    kp.wait_cycles = wait_cycles;
    if ((st = check_device(args->state)) != SSU_OK) return st;
    return launched(ssu::launch_onetoken(args->state_dtype, lanes, kp, batch, static_cast<cudaStream_t>(stream)));
}

ssu_status ssu_update_packed(const ssu_args *args, int64_t nseq, int64_t rows, const void *cu_seqlens,
                             int64_t steps, const void *num_accepted, int32_t meta_type,
                             const ssu_slot_table *read, const ssu_slot_table *dst, void *stream) {
    ssu::KParams kp;
    int lanes = 0;
    if (nseq < 0 || rows < 0) return fail(SSU_ERR_INVALID, "nseq and rows must not be negative");
    ssu_status st = prepare(args, rows, read, dst, &kp, &lanes);
    if (st != SSU_OK) return st;
    if ((cu_seqlens != nullptr || num_accepted != nullptr) && !valid_itype(meta_type))
        return fail(SSU_ERR_INVALID, "meta_type %d is not an ssu_itype", meta_type);
    if (cu_seqlens == nullptr) {
        if (steps <= 0) return fail(SSU_ERR_INVALID, "dense form (no cu_seqlens) needs steps > 0");
        if (rows != nseq * steps)
            return fail(SSU_ERR_INVALID, "dense form: rows (%lld) must equal nseq * steps (%lld)", (long long)rows,
                        (long long)(nseq * steps));
    }
    if (nseq == 0 || rows == 0) return ok();  // nothing to read or write
    if (nseq * kp.H * kp.ptiles > kMaxGrid) return fail(SSU_ERR_INVALID, "nseq * heads * dim tiles exceeds 2^31-1");
    if ((rows + nseq) > (int64_t(1) << 40) / (static_cast<int64_t>(kp.H) * kp.ptiles))
        return fail(SSU_ERR_INVALID, "(rows + nseq) * heads * dim tiles exceeds 2^40");
    kp.nseq = nseq;
    kp.rows = rows;
    kp.bulk_ops = packed_bulk_ops(args);
    kp.steps = cu_seqlens == nullptr ? steps : 0;
    kp.cu = cu_seqlens;
    kp.acc = num_accepted;
    kp.meta_is_i64 = meta_type == SSU_I64;
    if ((st = check_device(args->state)) != SSU_OK) return st;
    return launched(ssu::launch_packed(args->state_dtype, lanes, kp, static_cast<cudaStream_t>(stream)));
}

ssu_status ssu_replay_update(const ssu_args *args, int64_t batch, const ssu_slot_table *slots,
                             const ssu_replay_buffers *rb, void *stream) {
    ssu::KParams kp;
    int lanes = 0;
    if (batch < 0) return fail(SSU_ERR_INVALID, "batch is negative");
    ssu_status st = prepare(args, batch, slots, nullptr, &kp, &lanes);
    if (st != SSU_OK) return st;
    if (args->disable_state_update) return fail(SSU_ERR_INVALID, "disable_state_update is not defined for the replay step");
    if (rb == nullptr) return fail(SSU_ERR_INVALID, "replay buffers are NULL");
    if (rb->len < 1 || rb->len > ssu::kMaxReplayLen)
        return fail(SSU_ERR_UNSUPPORTED, "buffer length %lld is not supported (1..%d)", (long long)rb->len,
                    ssu::kMaxReplayLen);
    if (batch == 0) return ok();
    if (!rb->x || !rb->dt || !rb->B || !rb->count_in || !rb->count_out)
        return fail(SSU_ERR_INVALID, "replay buffers and counts must not be NULL");
    if (rb->count_out == rb->count_in) return fail(SSU_ERR_INVALID, "count_out must not alias count_in");
    if (batch * kp.H * kp.ptiles > kMaxGrid) return fail(SSU_ERR_INVALID, "batch * heads * dim tiles exceeds 2^31-1");
    kp.nseq = batch;
    kp.rows = batch;
    kp.rlen = static_cast<int32_t>(rb->len);
    kp.xbuf = rb->x;
    kp.dtbuf = rb->dt;
    kp.Bbuf = rb->B;
    kp.cnt_in = rb->count_in;
    kp.cnt_out = rb->count_out;
    {
        const int64_t io = args->io_dtype == SSU_F32 ? 4 : 2;
        const bool aligned = reinterpret_cast<uintptr_t>(rb->x) % 16 == 0 && reinterpret_cast<uintptr_t>(rb->dt) % 16 == 0 &&
                             reinterpret_cast<uintptr_t>(rb->B) % 16 == 0;
        kp.rbulk = aligned && (args->dim * io) % 16 == 0 && (args->dim * 4) % 16 == 0 && (args->dstate * io) % 16 == 0;
    }
    if (rb->reserved0 != 0) return fail(SSU_ERR_INVALID, "replay buffers: reserved0 must be 0");
    kp.shadow_fmt = rb->shadow_format;
    if (rb->shadow_format != SSU_SHADOW_NONE) {
        if (rb->shadow_format != SSU_SHADOW_F16 && rb->shadow_format != SSU_SHADOW_E4M3 &&
            rb->shadow_format != SSU_SHADOW_NVFP4)
            return fail(SSU_ERR_INVALID, "shadow_format %d is not an SSU_SHADOW_* value", rb->shadow_format);
        if (rb->shadow == nullptr || reinterpret_cast<uintptr_t>(rb->shadow) % 16 != 0)
            return fail(SSU_ERR_INVALID, "the read copy must be a 16-byte aligned device pointer");
        if (rb->shadow_format == SSU_SHADOW_E4M3) {
            if (rb->shadow_scale == nullptr || reinterpret_cast<uintptr_t>(rb->shadow_scale) % 16 != 0)
                return fail(SSU_ERR_INVALID, "E4M3 row scales must be a 16-byte aligned device pointer");
            if (args->dim % 4 != 0)
                return fail(SSU_ERR_UNSUPPORTED, "an E4M3 read copy needs dim to be a multiple of 4");
        }
        if (rb->shadow_format == SSU_SHADOW_NVFP4) {
            if (rb->shadow_scale == nullptr || reinterpret_cast<uintptr_t>(rb->shadow_scale) % 16 != 0)
                return fail(SSU_ERR_INVALID, "NVFP4 scale records must be a 16-byte aligned device pointer");
            if (args->dstate != 64 && args->dstate != 128 && args->dstate != 256)
                return fail(SSU_ERR_UNSUPPORTED, "an NVFP4 read copy needs dstate 64, 128 or 256");
        }
        kp.shadow = rb->shadow;
        kp.shadow_scale = rb->shadow_scale;
    }
    if ((st = check_device(args->state)) != SSU_OK) return st;
    return launched(ssu::launch_replay(args->state_dtype, lanes, kp, batch, static_cast<cudaStream_t>(stream)));
}

ssu_status ssu_replay_verify(const ssu_args *args, int64_t batch, int64_t ntok, const ssu_slot_table *slots,
                             const ssu_replay_buffers *rb, void *stream) {
    ssu::KParams kp;
    int lanes = 0;
    if (batch < 0) return fail(SSU_ERR_INVALID, "batch is negative");
    if (ntok < 1) return fail(SSU_ERR_INVALID, "ntok must be at least 1");
    ssu_status st = prepare(args, batch * ntok, slots, nullptr, &kp, &lanes);
    if (st != SSU_OK) return st;
    if (args->disable_state_update) return fail(SSU_ERR_INVALID, "disable_state_update is not defined for verification");
    if (rb == nullptr) return fail(SSU_ERR_INVALID, "replay buffers are NULL");
    if (rb->len < 1 || rb->len > ssu::kMaxReplayLen)
        return fail(SSU_ERR_UNSUPPORTED, "buffer length %lld is not supported (1..%d)", (long long)rb->len,
                    ssu::kMaxReplayLen);
    if (ntok > rb->len) return fail(SSU_ERR_INVALID, "ntok (%lld) exceeds the buffer length (%lld)", (long long)ntok,
                                    (long long)rb->len);
    if (rb->reserved0 != 0) return fail(SSU_ERR_INVALID, "replay buffers: reserved0 must be 0");
    if (rb->shadow_format != SSU_SHADOW_NONE)
        return fail(SSU_ERR_UNSUPPORTED, "verification does not read a low-precision copy");
    if (batch == 0) return ok();
    if (!rb->x || !rb->dt || !rb->B || !rb->count_in || !rb->count_out)
        return fail(SSU_ERR_INVALID, "replay buffers and counts must not be NULL");
    if (rb->count_out == rb->count_in) return fail(SSU_ERR_INVALID, "count_out must not alias count_in");
    if (args->heads > 65535 || batch > kMaxGrid || (args->dim + 63) / 64 > 65535)
        return fail(SSU_ERR_INVALID, "too many heads, sequences or dim rows for one launch");
    kp.nseq = batch;
    kp.rows = batch * ntok;
    kp.rlen = static_cast<int32_t>(rb->len);
    kp.xbuf = rb->x;
    kp.dtbuf = rb->dt;
    kp.Bbuf = rb->B;
    kp.cnt_in = rb->count_in;
    kp.cnt_out = rb->count_out;
    if ((st = check_device(args->state)) != SSU_OK) return st;
    return launched(ssu::launch_verify(args->state_dtype, kp, batch, static_cast<int>(ntok),
                                       static_cast<cudaStream_t>(stream)));
}

ssu_status ssu_batch_copy(const ssu_copy *copies, int64_t n, uint64_t max_bytes, int32_t *d_status,
                          void *stream) {
    if (n < 0) return fail(SSU_ERR_INVALID, "n is negative");
    if (n == 0 || max_bytes == 0) return ok();
    if (copies == nullptr) return fail(SSU_ERR_INVALID, "copies is NULL");
    if (reinterpret_cast<uintptr_t>(copies) % 8 != 0) return fail(SSU_ERR_INVALID, "copies must be 8-byte aligned");
    if (d_status != nullptr && reinterpret_cast<uintptr_t>(d_status) % 4 != 0)
        return fail(SSU_ERR_INVALID, "d_status must be 4-byte aligned");
    return launched(ssu::launch_copy(copies, n, max_bytes, d_status, static_cast<cudaStream_t>(stream)));
}

// Workspace carve-up of the SSD prefill: chunk states, prefix sums, dt',
// chunk decays, the largest |x| and dt' per (chunk, head); each part
// 256-byte aligned.
struct SsdWorkspace {
    uint64_t state, acs, dtp, dec, scl, total;
};
static SsdWorkspace ssd_workspace(uint64_t nchunks, uint64_t heads, uint64_t dim, uint64_t dstate,
                                  uint64_t chunk_size) {
    auto up = [](uint64_t v) { return (v + 255) / 256 * 256; };
    const uint64_t ch = nchunks * heads;
    SsdWorkspace w{};
    w.state = 0;
    w.acs = w.state + up(ch * dim * dstate * 4);
    w.dtp = w.acs + up(ch * chunk_size * 4);
    w.dec = w.dtp + up(ch * chunk_size * 4);
    w.scl = w.dec + up(ch * 4);
    w.total = w.scl + up(ch * 16);
    return w;
}

ssu_status ssu_ssd_workspace_size(int64_t nchunks, int64_t heads, int64_t groups, int64_t dim, int64_t dstate,
                                  int64_t chunk_size, uint64_t *bytes) {
    if (!bytes) return fail(SSU_ERR_INVALID, "bytes is NULL");
    if (nchunks < 0 || heads <= 0 || groups <= 0 || dim <= 0 || dstate <= 0 || chunk_size <= 0)
        return fail(SSU_ERR_INVALID, "sizes must be positive (nchunks >= 0)");
    *bytes = ssd_workspace(nchunks, heads, dim, dstate, chunk_size).total;
    return ok();
}

ssu_status ssu_ssd_prefill(const ssu_ssd_args *a, void *stream) {
    if (a == nullptr) return fail(SSU_ERR_INVALID, "args is NULL");
    if (a->tokens < 0 || a->nseq < 0 || a->nchunks < 0) return fail(SSU_ERR_INVALID, "negative sizes");
    if (a->heads <= 0 || a->groups <= 0 || a->heads % a->groups != 0)
        return fail(SSU_ERR_INVALID, "heads (%lld) must be a positive multiple of groups (%lld)", (long long)a->heads,
                    (long long)a->groups);
    if (a->io_dtype != SSU_BF16) return fail(SSU_ERR_UNSUPPORTED, "the SSD prefill takes bf16 x, z, B, C and y");
    if (!valid_dtype(a->dt_dtype) || !valid_dtype(a->state_dtype)) return fail(SSU_ERR_INVALID, "bad dtype");
    if (!valid_itype(a->meta_type)) return fail(SSU_ERR_INVALID, "meta_type %d is not an ssu_itype", a->meta_type);
    if (a->dim != 64) return fail(SSU_ERR_UNSUPPORTED, "the SSD prefill supports dim 64 (got %lld)", (long long)a->dim);
    if (a->dstate != 64 && a->dstate != 128)
        return fail(SSU_ERR_UNSUPPORTED, "the SSD prefill supports dstate 64 or 128 (got %lld)", (long long)a->dstate);
    if (a->chunk_size != 64 && a->chunk_size != 128 && a->chunk_size != 256)
        return fail(SSU_ERR_UNSUPPORTED, "chunk_size %lld is not supported (64, 128, 256)", (long long)a->chunk_size);
    if (!(a->dt_min <= a->dt_max)) return fail(SSU_ERR_INVALID, "dt_limit must satisfy min <= max");
    if (a->nchunks == 0 || a->tokens == 0) return ok();
    if (a->nchunks > 65535 || a->heads > 65535) return fail(SSU_ERR_INVALID, "more than 65535 chunks or heads");
    if (!a->x || !a->dt || !a->B || !a->C || !a->A || !a->cu_chunk_seqlens || !a->seq_idx || !a->y || !a->states ||
        (!a->return_intermediate && !a->last_chunk_indices) || !a->workspace)
        return fail(SSU_ERR_INVALID, "a required pointer is NULL");
    const void *aligned[] = {a->x, a->B, a->C, a->y, a->states, a->workspace, a->z, a->initial_states};
    for (const void *q : aligned)
        if (reinterpret_cast<uintptr_t>(q) % 16 != 0) return fail(SSU_ERR_INVALID, "tensors must be 16-byte aligned");
    const SsdWorkspace wl = ssd_workspace(a->nchunks, a->heads, a->dim, a->dstate, a->chunk_size);
    const uint64_t need = wl.total;
    if (a->workspace_bytes < need)
        return fail(SSU_ERR_INVALID, "workspace of %lld bytes is smaller than the %lld needed",
                    (long long)a->workspace_bytes, (long long)need);
    ssu::SsdParams p{};
    p.tokens = a->tokens;
    p.nchunks = a->nchunks;
    p.nseq = a->nseq;
    p.H = static_cast<int32_t>(a->heads);
    p.G = static_cast<int32_t>(a->groups);
    p.hpg = static_cast<int32_t>(a->heads / a->groups);
    p.P = static_cast<int32_t>(a->dim);
    p.N = static_cast<int32_t>(a->dstate);
    p.Q = static_cast<int32_t>(a->chunk_size);
    p.dt_dtype = a->dt_dtype;
    p.state_dtype = a->state_dtype;
    p.softplus = a->dt_softplus != 0;
    p.intermediate = a->return_intermediate != 0;
    p.meta_i64 = a->meta_type == SSU_I64;
    p.dt_lo = a->dt_min;
    p.dt_hi = a->dt_max;
    p.x = a->x, p.dt = a->dt, p.B = a->B, p.C = a->C, p.z = a->z;
    p.A = a->A, p.D = a->D, p.dt_bias = a->dt_bias;
    p.cu_chunk = a->cu_chunk_seqlens, p.seq_idx = a->seq_idx, p.last_chunk = a->last_chunk_indices;
    p.init = a->initial_states;
    p.y = a->y;
    p.states = a->states;
    p.status = a->d_status;
    {
        unsigned char *w = static_cast<unsigned char *>(a->workspace);
        p.ws_state = reinterpret_cast<float *>(w + wl.state);
        p.ws_acs = reinterpret_cast<float *>(w + wl.acs);
        p.ws_dtp = reinterpret_cast<float *>(w + wl.dtp);
        p.ws_dec = reinterpret_cast<float *>(w + wl.dec);
        p.ws_scl = reinterpret_cast<float *>(w + wl.scl);
    }
    return launched(ssu::launch_ssd(p, static_cast<cudaStream_t>(stream)));
}

ssu_status ssu_ssd_prefill_static(const ssu_ssd_args *args, void *stream) {
    if (args == nullptr) return fail(SSU_ERR_INVALID, "args is NULL");
    if (args->workspace != nullptr || args->workspace_bytes != 0)
        return fail(SSU_ERR_INVALID, "workspace must be NULL and workspace_bytes 0 (the library's scratch is used)");
    uint64_t need = 0;
    const ssu_status st = ssu_ssd_workspace_size(args->nchunks, args->heads, args->groups, args->dim, args->dstate,
                                                 args->chunk_size, &need);
    if (st != SSU_OK) return st;
    if (need > ssu::kSsdStaticScratchBytes)
        return fail(SSU_ERR_INVALID, "the call needs %llu bytes of workspace; the library's scratch holds %llu",
                    (unsigned long long)need, (unsigned long long)ssu::kSsdStaticScratchBytes);
    if (args->nchunks == 0 || args->tokens == 0) return ssu_ssd_prefill(args, stream);
    void *scratch = nullptr;
    const cudaError_t e = ssu::ssd_static_scratch(&scratch);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "looking up the scratch failed: %s", cudaGetErrorString(e));
    ssu_ssd_args a = *args;
    a.workspace = scratch;
    a.workspace_bytes = ssu::kSsdStaticScratchBytes;
    return ssu_ssd_prefill(&a, stream);
}

ssu_status ssu_shadow_refresh(const void *state, int32_t state_dtype, int64_t rows, int64_t dstate,
                              int32_t format, void *shadow, float *scale, void *stream) {
    if (!valid_dtype(state_dtype)) return fail(SSU_ERR_INVALID, "state_dtype %d is not an ssu_dtype", state_dtype);
    if (format != SSU_SHADOW_F16 && format != SSU_SHADOW_E4M3 && format != SSU_SHADOW_NVFP4)
        return fail(SSU_ERR_INVALID, "format %d is not SSU_SHADOW_F16, SSU_SHADOW_E4M3 or SSU_SHADOW_NVFP4", format);
    if (rows < 0 || dstate <= 0 || dstate > 4096) return fail(SSU_ERR_INVALID, "rows must be >= 0, dstate in [1, 4096]");
    if (format == SSU_SHADOW_NVFP4 && dstate % 32 != 0)
        return fail(SSU_ERR_UNSUPPORTED, "an NVFP4 read copy needs dstate to be a multiple of 32");
    if (rows == 0) return ok();
    if (!state || !shadow || (format != SSU_SHADOW_F16 && !scale))
        return fail(SSU_ERR_INVALID, "state, shadow (and scale for E4M3 and NVFP4) must not be NULL");
    return launched(ssu::launch_shadow_refresh(state, state_dtype, rows, static_cast<int>(dstate), format, shadow,
                                               scale, static_cast<cudaStream_t>(stream)));
}

ssu_status ssu_prewarm(int32_t state_dtype, int32_t io_dtype, int32_t dt_dtype, int64_t heads, int64_t dim,
                       int64_t dstate, int64_t groups, int32_t packed) {
    int lanes = 0;
    ssu_status st = check_shape(state_dtype, io_dtype, dt_dtype, heads, dim, dstate, groups, &lanes);
    if (st != SSU_OK) return st;
    cudaError_t e = packed ? ssu::prewarm_packed(state_dtype, lanes) : ssu::prewarm_onetoken(state_dtype, lanes);
    if (e != cudaSuccess) return fail(SSU_ERR_CUDA, "loading the kernel failed: %s", cudaGetErrorString(e));
    return ok();
}

const char *ssu_last_error(void) { return g_err; }

}  // extern "C"
