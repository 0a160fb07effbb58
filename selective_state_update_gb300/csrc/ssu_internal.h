// ssu_internal.h -- parameters shared by the host layer and the kernels of
// libssu.  Not part of the public ABI (that is include/ssu.h).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace ssu {

// Each thread holds kRowsPerThread rows x kElemsPerThread dstate elements.
constexpr int kRowsPerThread = 4;
// Rows of one (head, dim-tile) work unit: kTileRows dim rows of one head of
// one sequence.
constexpr int kTileRows = 16 * kRowsPerThread;
constexpr int kElemsPerThread = 16;
// Row slots per CTA: kTileRows / kRowsPerThread.  A CTA has
// kRowSlots * L threads, L = dstate / kElemsPerThread lanes per row.
constexpr int kRowSlots = kTileRows / kRowsPerThread;
// How many of a thread's rows the one-token compute loop keeps in flight at
// once (more rows: more loads in flight, more registers, fewer resident CTAs).
constexpr int kOnetokenUnroll = 2;

struct SlotTab {
    const void *entries;  // nullptr: no table
    int64_t s0, s1, extent;
    int32_t is_i64;
    int32_t per_row;
};

struct KParams {
    // shape
    int64_t slots;
    int32_t H, P, N, G, heads_per_group, ptiles;
    // dtypes (ssu_dtype values) of the small operands
    int32_t io_dtype, dt_dtype;
    int32_t softplus, disable;
    int64_t pad;
    // operands
    void *state;
    const void *x, *dt, *B, *C, *z;
    const float *A, *D, *dt_bias;
    void *y;
    int64_t xs[3], dts[3], Bs[3], Cs[3], zs[3], ys[3];
    // slot tables (rd.entries == nullptr: slot b; wr.entries == nullptr: use rd)
    SlotTab rd, wr;
    // packed layout
    int64_t nseq, rows, steps;  // steps > 0 with cu == nullptr: dense form
    const void *cu, *acc;
    int32_t meta_is_i64;
    int32_t *status;
    // checkpoint + buffer form (ssu_replay_update)
    int32_t rlen;
    void *xbuf;
    float *dtbuf;
    void *Bbuf;
    const int32_t *cnt_in;
    int32_t *cnt_out;
    int32_t rbulk;  // buffer rows are 16-byte aligned: stage them with bulk copies
    // low-precision read copy of the checkpoints (kShadow*)
    int32_t shadow_fmt;
    void *shadow;
    float *shadow_scale;
    // bounded waits: SM clock cycles before a wait gives up
    int64_t wait_cycles;
    // self-test of the exit path (ssu_selftest_timeout): the one-token
    // producer skips the copy and the arrival of this unit (-1: none)
    int64_t withhold_unit;
    // packed kernel: which small operands arrive by bulk copies (kBulk* bits)
    int32_t bulk_ops;
};

enum : int32_t { kBulkBC = 1, kBulkXZ = 2, kBulkDT = 4 };

// SM clock cycles a bounded wait allows by default (about a second).
constexpr int64_t kDefaultWaitCycles = 2000000000LL;

enum : int32_t { kShadowNone = 0, kShadowF16 = 1, kShadowE4M3 = 2, kShadowNVFP4 = 3 };

// Launchers (one translation unit per kernel).  `lanes` = dstate / 16.
cudaError_t launch_onetoken(int state_dtype, int lanes, const KParams &p, int64_t batch,
                            cudaStream_t stream);
cudaError_t launch_packed(int state_dtype, int lanes, const KParams &p, cudaStream_t stream);
// The packed kernel for long sequences (one CTA per unit), which
// launch_packed picks when rows >= kLongRowsPerSeq * nseq.
constexpr int64_t kLongRowsPerSeq = 6;
cudaError_t launch_packed_long(int state_dtype, int lanes, const KParams &p, cudaStream_t stream);
cudaError_t prewarm_packed_long(int state_dtype, int lanes);
// Load the kernel's module and read its attributes (no launch).
cudaError_t prewarm_onetoken(int state_dtype, int lanes);
cudaError_t prewarm_packed(int state_dtype, int lanes);
cudaError_t launch_replay(int state_dtype, int lanes, const KParams &p, int64_t batch, cudaStream_t stream);

// The read copy of `rows` state rows (ssu_shadow_refresh).
cudaError_t launch_shadow_refresh(const void *state, int state_dtype, int64_t rows, int dstate, int format,
                                  void *shadow, float *scale, cudaStream_t stream);
// Batched copies (ssu_batch_copy): `copies` device [n] {src, dst, bytes}.
cudaError_t launch_copy(const void *copies, int64_t n, uint64_t max_bytes, int32_t *status, cudaStream_t stream);

// Largest buffer length of the checkpoint + buffer form.
constexpr int kMaxReplayLen = 32;

}  // namespace ssu
