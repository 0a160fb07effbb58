/*
 * ssu.h -- libssu: the Mamba-2 selective state update (SSU) on NVIDIA GB300
 * (sm_103a), behind a plain C ABI.
 *
 * What one call computes (MATE documentation, page "Mamba / SSU": intro
 * paragraph, "SSU at a glance", API reference of selective_state_update; the
 * recurrence as written in the article "ReplaySSM: Cache SSM Inputs, Not
 * State", section 三个瓶颈).  For every token row r of a sequence, every head h
 * and every dim row p, with g = h / (heads / groups):
 *
 *     dt'  = dt[r,h,p] (+ dt_bias[h]);  dt' = softplus(dt') if dt_softplus
 *     dA   = exp(A[h] * dt')
 *     S[n] = S[n] * dA + dt' * x[r,h,p] * B[r,g,n]          (n < dstate)
 *     y[r,h,p] = sum_n S[n] * C[r,g,n] + D[h] * x[r,h,p]
 *     y[r,h,p] *= z / (1 + exp(-z)),  z = z[r,h,p]            (when z given)
 *
 * S is one row of the state pool, read from the sequence's read slot, carried
 * in fp32 across the sequence's tokens, and published (rounded to nearest
 * even into the state dtype) to each token's destination slot.  y is
 * computed in fp32 and rounded to nearest even into the io dtype.
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device pointers on the current device
 *    (a state pool on another device is rejected with SSU_ERR_INVALID);
 *    the caller owns every buffer.  The library allocates no device memory,
 *    copies nothing between host and device, and never synchronizes: one
 *    call is one kernel launch on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  After ssu_prewarm the calls may be captured in
 *    a CUDA graph.
 *  - Host-detectable errors return a status, leave a message for
 *    ssu_last_error(), and launch nothing.
 *  - Errors only the device can see (a slot outside [0, slots) that is not
 *    the pad id, a table entry outside the table, malformed cu_seqlens)
 *    never trap: the kernel ORs an SSU_DEV_* bit into *d_status (when
 *    d_status is not NULL) and skips the affected (sequence, head) unit:
 *    none of its state rows and none of its y rows are written.
 *  - Preconditions not checked: buffers do not overlap except where stated
 *    (the pool may be read and written through the same slot); no sequence
 *    writes a slot that another sequence of the same call reads or writes
 *    (the result would depend on scheduling); y does not alias any input.
 */
#ifndef SSU_H
#define SSU_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSU_OK = 0,
    SSU_ERR_INVALID = 1,      /* an argument check failed (Python: ValueError)            */
    SSU_ERR_UNSUPPORTED = 2,  /* the caller asked for something not implemented
                                 (Python: NotImplementedError)                             */
    SSU_ERR_CUDA = 3          /* a CUDA runtime call failed (launch or attribute query)    */
} ssu_status;

/* Element types.  The state pool may be any of the three (MATE "Mamba / SSU",
 * SSU at a glance, row State).  x, z, y, B and C share one io type (row B / C:
 * "with the x dtype"; row Output: "in the x dtype").  A, D and dt_bias are
 * always fp32 (row A / D / dt_bias). */
typedef enum { SSU_F32 = 0, SSU_F16 = 1, SSU_BF16 = 2 } ssu_dtype;

/* Integer types of slot tables, cu_seqlens and num_accepted_tokens. */
typedef enum { SSU_I32 = 0, SSU_I64 = 1 } ssu_itype;

/* How a slot table is addressed for (sequence b, step t).
 *  SSU_SLOTS_STRIDED: entry = b*s0 + t*s1.  This is the page's rule (Slot
 *    semantics): a flat [n] table is addressed as [n, 1] (s0 = s1 = 1, entry
 *    b + t) and a contiguous 2-D [seqs, steps] table as b*steps + t.
 *  SSU_SLOTS_PER_ROW: entry = cu_seqlens[b] + t, one entry per packed row
 *    (the flat form vLLM's MTP decode passes).  The two agree whenever the
 *    strided form is free of collisions: one sequence per call, or every
 *    sequence of length 1 with no empties.  With several sequences longer
 *    than one token, the strided flat form makes neighbouring sequences share
 *    entries and is only meaningful with disable_state_update. */
typedef enum { SSU_SLOTS_STRIDED = 0, SSU_SLOTS_PER_ROW = 1 } ssu_slot_mode;

typedef struct ssu_slot_table {
    const void *entries;  /* device pointer to `type` entries; NULL = no table        */
    int32_t type;         /* ssu_itype                                                  */
    int32_t mode;         /* ssu_slot_mode                                              */
    int64_t s0, s1;       /* strides in entries (SSU_SLOTS_STRIDED)                     */
    int64_t extent;       /* entries [0, extent) may be addressed; others set
                             SSU_DEV_BAD_ENTRY                                          */
} ssu_slot_table;

/* Bits ORed into *d_status by the kernels. */
#define SSU_DEV_BAD_SLOT   0x1  /* slot not in [0, slots) and not pad_slot_id       */
#define SSU_DEV_BAD_ENTRY  0x2  /* table entry index outside [0, extent), or a
                                   per-row seed step past its sequence's rows      */
#define SSU_DEV_BAD_SEQLEN 0x4  /* cu_seqlens decreasing, negative or past `rows`   */
#define SSU_DEV_TIMEOUT    0x8  /* an asynchronous state copy did not complete in
                                   about a second; the unit was skipped           */
#define SSU_DEV_BAD_COUNT  0x10 /* replay / verify: a buffered count outside [0, L) */
#define SSU_DEV_BAD_COPY   0x20 /* ssu_batch_copy: a copy longer than max_bytes      */

/* Arguments of the MATE signature that this library does not implement.  Set
 * the bit when the caller passed the argument; the call then fails with
 * SSU_ERR_UNSUPPORTED instead of silently narrowing the semantics (the page
 * raises NotImplementedError for rand_seed, "Stochastic rounding" row). */
#define SSU_UNSUP_RAND_SEED          0x01  /* stochastic rounding                     */
#define SSU_UNSUP_STATE_SCALE        0x02  /* quantised state scales                   */
#define SSU_UNSUP_INTERMEDIATE       0x04  /* intermediate_states_buffer / indices / scales */
#define SSU_UNSUP_CACHE_STEPS        0x08  /* cache_steps != 0                         */
#define SSU_UNSUP_ALGORITHM          0x10  /* algorithm / backend other than "auto"   */

/* Everything both update entry points share.  Strides are in elements. */
typedef struct ssu_args {
    int64_t slots, heads, dim, dstate, groups;
    int32_t state_dtype;          /* ssu_dtype of the pool                                   */
    int32_t io_dtype;             /* ssu_dtype of x, z, y, B, C (SSU_BF16 or SSU_F16 or SSU_F32) */
    int32_t dt_dtype;             /* ssu_dtype of dt                                         */
    int32_t dt_softplus;          /* nonzero: dt' = softplus(dt + dt_bias)                   */
    int32_t disable_state_update; /* nonzero: the pool is not written (y still is)           */
    int32_t reserved0;            /* must be 0                                               */
    int64_t pad_slot_id;          /* slot id that reads as a zero state and is never written */
    void *state;                  /* device [slots, heads, dim, dstate], contiguous, 16-byte
                                     aligned; read and written in place                       */
    const void *x;                /* device [rows, heads, dim] io_dtype                       */
    const void *dt;               /* device [rows, heads, dim] dt_dtype; dt_stride[2] == 0
                                     gives one step per head broadcast over dim              */
    const void *B, *C;            /* device [rows, groups, dstate] io_dtype                   */
    const void *z;                /* device [rows, heads, dim] io_dtype, or NULL (no gate)     */
    const float *A;               /* device [heads]                                          */
    const float *D;               /* device [heads] or NULL (no skip term)                   */
    const float *dt_bias;         /* device [heads] or NULL                                  */
    void *y;                      /* device [rows, heads, dim] io_dtype, output              */
    int64_t x_stride[3], dt_stride[3], B_stride[3], C_stride[3], z_stride[3], y_stride[3];
    int32_t *d_status;            /* device int32 or NULL; SSU_DEV_* bits are ORed in        */
    uint32_t unsupported;         /* SSU_UNSUP_* bits; nonzero => SSU_ERR_UNSUPPORTED         */
} ssu_args;

/*
 * One decode token per sequence: sequence b is row b (x, dt, z, y are
 * [batch, heads, dim]; B, C are [batch, groups, dstate]).
 * MATE "Mamba / SSU": intro paragraph (the one-token kernel); SSU at a glance,
 * rows Sequence layout, State, Slot semantics.
 *
 *   read  NULL or read->entries NULL: sequence b reads slot b.  Otherwise the
 *         slot at entry (b, 0) of the table (the mode is ignored: a one-token
 *         call has cu_seqlens[b] = b).
 *   dst   NULL or dst->entries NULL: the state is written back through the
 *         read table (or to slot b without one).  Otherwise to entry (b, 0).
 *   A read of pad_slot_id starts from zeros; a write to it is skipped.
 * batch == 0 launches nothing and returns SSU_OK; the row operands may then
 * be NULL.
 */
ssu_status ssu_update_onetoken(const ssu_args *args, int64_t batch,
                               const ssu_slot_table *read, const ssu_slot_table *dst,
                               void *stream);

/*
 * Packed variable-length / multi-token (MTP) decode: `rows` packed rows split
 * into `nseq` sequences.  MATE "Mamba / SSU": SSU at a glance, rows Sequence
 * layout, Slot semantics, Variable-length and MTP decode; Graph capture
 * (single launch, no host/device scalar copies).
 *
 *   cu_seqlens   device [nseq + 1] of meta_type: sequence b owns rows
 *                [cu_seqlens[b], cu_seqlens[b+1]).  NULL selects the dense
 *                form: every sequence is `steps` rows long (rows = nseq*steps),
 *                i.e. x as [nseq, steps, heads, dim] flattened.
 *   num_accepted device [nseq] of meta_type or NULL.  The read slot of
 *                sequence b is at step max(num_accepted[b] - 1, 0) (step 0
 *                without the array).  With a SSU_SLOTS_PER_ROW read table
 *                that step must be one of the sequence's own rows (below
 *                its length): a later one would name another sequence's
 *                entry, so the sequence sets SSU_DEV_BAD_ENTRY and is
 *                skipped.
 *   read, dst    slot tables addressed per their mode (see ssu_slot_mode).
 *                No read table: sequence b reads and writes slot b (every
 *                token overwrites it; the last token's state remains).  No
 *                destination table: token t publishes through the read
 *                table's entry (b, t).
 * Every token publishes its state to its own destination slot unless that
 * slot is pad_slot_id or disable_state_update is set.  Empty sequences are
 * skipped.  The state carried between the tokens of a sequence stays in
 * fp32; only the published copies are rounded.  A sequence may overwrite its
 * own read slot (the read happens first).
 * nseq == 0 or rows == 0 launches nothing and returns SSU_OK (every
 * sequence is then empty; cu_seqlens is not read).  With rows == 0 the row
 * operands (x, dt, B, C, z, y) may be NULL.
 */
ssu_status ssu_update_packed(const ssu_args *args, int64_t nseq, int64_t rows,
                             const void *cu_seqlens, int64_t steps,
                             const void *num_accepted, int32_t meta_type,
                             const ssu_slot_table *read, const ssu_slot_table *dst,
                             void *stream);

/*
 * The decode state of a slot kept as a checkpoint plus a buffer of the inputs
 * of the steps since the last fold (article "ReplaySSM: Cache SSM Inputs, Not
 * State", sections 核心做法 and 数据与边界: the checkpoint is read every step
 * but written once every L steps).  For each slot s the buffer holds up to
 * L - 1 entries j (the inputs of one past step): x and B as given, and the
 * processed step dt' = softplus(dt + dt_bias) in fp32, so that a fold repeats
 * exactly the updates the plain step would have made.
 */
typedef struct ssu_replay_buffers {
    int64_t len;               /* L, 1 <= L <= 32                                         */
    void *x;                   /* device [slots, L, heads, dim] io_dtype, contiguous       */
    float *dt;                 /* device [slots, L, heads, dim] fp32, contiguous           */
    void *B;                   /* device [slots, L, groups, dstate] io_dtype, contiguous   */
    const int32_t *count_in;   /* device [batch]: entries buffered for sequence b          */
    int32_t *count_out;        /* device [batch]: entries after the call (written); must
                                  not alias count_in                                      */
    /* Optional low-precision read copy of the checkpoints (article
     * "ReplaySSM", section 低精度读写分离): steps that do not fold read it
     * instead of the checkpoint, a fold rewrites it from the new checkpoint
     * (as ssu_shadow_refresh would).  It never feeds the recurrence. */
    int32_t shadow_format;     /* SSU_SHADOW_NONE, _F16, _E4M3 or _NVFP4                  */
    int32_t reserved0;         /* must be 0                                               */
    void *shadow;              /* device [slots, heads, dim, dstate]: fp16 values or E4M3
                                  codes (one byte); NVFP4: [slots, heads, dim, dstate / 2]
                                  bytes of two E2M1 codes; 16-byte aligned                */
    float *shadow_scale;       /* device, 16-byte aligned: E4M3 [slots, heads, dim] fp32
                                  row scales; NVFP4 [slots, heads, dim,
                                  SSU_NVFP4_SCALE_WORDS(dstate)] scale records; unused
                                  for F16                                                 */
} ssu_replay_buffers;

/* Formats of the read copy.  E4M3 is OCP FP8 E4M3 (bias 7, 3 fraction bits,
 * no infinities, largest 448) with one fp32 scale per state row: the row's
 * largest magnitude amax maps to 448, code = E4M3(v * 448 / amax) rounded to
 * nearest even and clamped to +-448, and scale = amax / 448 in fp32 (1, with
 * zero codes, for an all-zero row); the value read is E4M3(code) * scale.
 * The kernels form the quotient in fp32 as v * (448 / amax), so a code can
 * sit one step from the exactly rounded one where v * 448 / amax lies within
 * about 2^-22 (relative) of a midpoint between two E4M3 values.  F16 is
 * binary16, round to nearest even. */
#define SSU_SHADOW_NONE 0
#define SSU_SHADOW_F16  1
#define SSU_SHADOW_E4M3 2
/* NVFP4 (the article's headline format for the copy): FP4 E2M1 codes (sign,
 * 2 exponent bits with bias 1, 1 fraction bit: magnitudes 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6), two a byte with the even element in the low nibble, scaled on
 * two levels: per block of 16 elements an E4M3 code of (block amax) / (6 s),
 * and per state row an fp32 s = amax / (6 * 448) (1, with zero codes, for an
 * all-zero row); element code = E2M1(v / (block scale * s)), the quotients in
 * fp32, roundings to nearest even, saturating.  The value read is
 * E2M1(code) * E4M3(block code) * s.  Each row's record in shadow_scale holds
 * s, then the dstate / 16 block codes as bytes, padded to a multiple of 16
 * bytes (SSU_NVFP4_SCALE_WORDS floats).  A code or block code can sit one step
 * from the exactly rounded one where its quotient lies within about 2^-21
 * (relative) of a midpoint.  Replay steps take it at dstate 64, 128 and 256;
 * ssu_shadow_refresh at any multiple of 32. */
#define SSU_SHADOW_NVFP4 3
#define SSU_NVFP4_SCALE_WORDS(dstate) ((4 + (dstate) / 16 + 15) / 16 * 4)

/*
 * One decode token per sequence on the checkpoint + buffer form of the state
 * (article "ReplaySSM: Cache SSM Inputs, Not State", section 核心做法).
 * args->state is the checkpoint pool; x, dt, z, B, C, y are one row per
 * sequence as for ssu_update_onetoken; `slots` gives sequence b's slot at
 * entry b (NULL: slot b); checkpoint and buffers are read and written through
 * that one slot.  With c = count_in[b]:
 *   c + 1 <  L  y is read out of checkpoint and buffer without forming the
 *               state, y = (gamma S_ckpt.C + sum_j gamma_j dt'_j x_j (B_j.C)
 *               + D x) * silu(z), gamma products of exp(A dt') from the entry
 *               after j to the current token; the current token is appended
 *               as entry c and count_out[b] = c + 1; the checkpoint is not
 *               written;
 *   c + 1 == L  the buffer is folded into the checkpoint (the entries, then
 *               the current token, in order, carried in fp32), the state is
 *               written back once, y is read out of it, count_out[b] = 0.
 * L = 1 is exactly ssu_update_onetoken with the destination equal to the read
 * slot.  A pad slot reads as a zero state with no history: y from the current
 * token alone, nothing written, count_out[b] = 0.  A count outside [0, L) sets
 * SSU_DEV_BAD_COUNT and skips the sequence.  disable_state_update must be 0.
 * With a read copy (rb->shadow_format != SSU_SHADOW_NONE) the S_ckpt.C of a
 * step that does not fold comes from the copy; dim must be a multiple of 4
 * for E4M3 (row scales move in 16-byte pieces).
 * The dstate and dtype rules of ssu_update_onetoken apply.  batch == 0
 * launches nothing.
 */
ssu_status ssu_replay_update(const ssu_args *args, int64_t batch, const ssu_slot_table *slots,
                             const ssu_replay_buffers *rb, void *stream);

/*
 * Speculative decoding on the checkpoint + buffer form (article "ReplaySSM:
 * Cache SSM Inputs, Not State", section 投机解码回滚).  Each of `batch`
 * sequences brings `ntok` = T draft tokens: the row operands of `args` (x, dt,
 * z, B, C, y) hold row b * T + k for draft k of sequence b.  With c =
 * count_in[b] committed entries in the sequence's buffer:
 *   c + 2T >= L  the committed entries are first folded into the checkpoint
 *                (written once) and c becomes 0 -- the flush one window early,
 *                so that the next step finds T free entries;
 *   then         the drafts are appended as entries c .. c+T-1 (x and B keep
 *                their bits, dt' = softplus?(dt + dt_bias) in fp32) and draft
 *                k's y is the output after the checkpoint (as stored), the
 *                committed entries and drafts 0 .. k in order (causal mask),
 *                every step with its dt' as stored;
 *   count_out[b] = c: nothing is committed.  Accepting the first a drafts is
 *                setting the count to count_out[b] + a (later entries are
 *                overwritten by later appends); no state is restored.
 * A pad slot reads as a zero state with no history: y from the drafts alone,
 * nothing written, count_out[b] = 0.  A count outside [0, L) sets
 * SSU_DEV_BAD_COUNT and skips the sequence; bad table entries and slots set
 * their bits as for ssu_replay_update.  1 <= T <= L; no read copy
 * (rb->shadow_format must be SSU_SHADOW_NONE); disable_state_update must be
 * 0; the dstate and dtype rules of ssu_update_onetoken apply.  Two kernel
 * launches on `stream`; batch == 0 launches nothing.
 */
ssu_status ssu_replay_verify(const ssu_args *args, int64_t batch, int64_t ntok, const ssu_slot_table *slots,
                             const ssu_replay_buffers *rb, void *stream);

/*
 * Packed variable-length SSD prefill (MATE documentation, page "Mamba / SSU",
 * section "SSD packed prefill" and the API reference of
 * ssd_combined_fwd_varlen).  For every token t of a packed batch, head h,
 * dim row p, g = h / (heads / groups):
 *     dt'  = clamp(softplus?(dt[t,h] + dt_bias[h]), dt_min, dt_max)
 *     S[n] = S[n] exp(A[h] dt') + dt' x[t,h,p] B[t,g,n]
 *     y[t,h,p] = (sum_n S[n] C[t,g,n] + D[h] x[t,h,p]) * silu(z[t,h,p])
 * evaluated chunk by chunk (cumulative decays, chunk states, state passing,
 * C . B^T, chunk scan).  Chunk c covers tokens [cu_chunk_seqlens[c],
 * cu_chunk_seqlens[c+1]) (at most chunk_size tokens); chunk c opens a
 * sequence when c == 0 or seq_idx[c] != seq_idx[c-1] -- seq_idx, not
 * last_chunk_indices, decides -- and then starts from
 * initial_states[seq_idx[c]] (zero without initial states); otherwise it
 * continues from the previous chunk's state.  `states` receives the state at
 * the end of every chunk ([nchunks, heads, dim, dstate]) when
 * return_intermediate is set, otherwise the state at the end of chunk
 * last_chunk_indices[b] for every sequence b ([nseq, heads, dim, dstate]),
 * in state_dtype.  Implemented: x, z, B, C and y bf16, contiguous; dt fp32 /
 * fp16 / bf16 [tokens, heads]; dim 64; dstate 64 or 128; chunk_size 64, 128
 * or 256 (others return SSU_ERR_UNSUPPORTED).  The contractions run on the
 * tensor cores with fp32 accumulation: C . B^T with bf16 operands; the chunk
 * states with a two-part bf16 split of the decay-weighted x; the entering
 * state's term with a two-part bf16 split of the state; the causal weights
 * (C . B^T) exp(cs_t - cs_s) dt'_s times x with fp16 operands (x is exact in
 * fp16 where bf16 values lie in fp16's normal range, about 6.1e-5 to 65504
 * in magnitude).  `workspace` is
 * caller-owned device memory of at least ssu_ssd_workspace_size() bytes,
 * 256-byte aligned; its contents need no initialisation.  Malformed chunks
 * (negative, decreasing, longer than chunk_size or past `tokens`) set
 * SSU_DEV_BAD_SEQLEN and produce no y; a seq_idx outside [0, nseq), or (without
 * return_intermediate) a last_chunk_indices entry outside [0, nchunks), sets
 * SSU_DEV_BAD_ENTRY and leaves the states it concerns unwritten.  Host-side
 * errors (NULL pointers, unaligned tensors, a short workspace) return
 * SSU_ERR_INVALID before anything is launched.
 */
typedef struct ssu_ssd_args {
    int64_t tokens, heads, dim, dstate, groups, nseq, nchunks, chunk_size;
    int32_t io_dtype;              /* SSU_BF16                                              */
    int32_t dt_dtype, state_dtype; /* ssu_dtype                                             */
    int32_t meta_type;             /* SSU_I32 / SSU_I64: cu_chunk_seqlens, seq_idx, last... */
    int32_t dt_softplus;
    int32_t return_intermediate;
    float dt_min, dt_max;          /* dt_limit; (0, +inf) leaves dt' unclamped above        */
    const void *x;                 /* device [tokens, heads, dim]                           */
    const void *dt;                /* device [tokens, heads]                                */
    const void *B, *C;             /* device [tokens, groups, dstate]                       */
    const void *z;                 /* device [tokens, heads, dim] or NULL                   */
    const float *A, *D, *dt_bias;  /* device [heads] fp32; D and dt_bias may be NULL        */
    const void *cu_chunk_seqlens;  /* device [nchunks + 1]                                  */
    const void *seq_idx;           /* device [nchunks]                                      */
    const void *last_chunk_indices;/* device [nseq]                                         */
    const void *initial_states;    /* device [nseq, heads, dim, dstate] state_dtype, or NULL */
    void *y;                       /* device [tokens, heads, dim] (out)                     */
    void *states;                  /* device, see above (out)                               */
    void *workspace;
    uint64_t workspace_bytes;
    int32_t *d_status;             /* device int32 or NULL                                  */
} ssu_ssd_args;

/* Workspace ssu_ssd_prefill needs for these sizes (bytes, into *bytes):
 * the chunk states (fp32; later the entering states as bf16 high and low
 * parts in their place), per-chunk prefix sums, dt' and decays, and the
 * largest |x| and dt' of every (chunk, head).  `groups`
 * is checked (positive) but takes no part in the size. */
ssu_status ssu_ssd_workspace_size(int64_t nchunks, int64_t heads, int64_t groups, int64_t dim, int64_t dstate,
                                  int64_t chunk_size, uint64_t *bytes);

/* One packed SSD prefill call: three kernel launches on `stream` (at most
 * 65535 chunks and 65535 heads per call). */
ssu_status ssu_ssd_prefill(const ssu_ssd_args *args, void *stream);

/*
 * ssu_ssd_prefill on a workspace the library owns, for callers that hold no
 * device memory of their own for it; the pages have no counterpart (their
 * wrapper caches a workspace it allocates).  args->workspace must be NULL and
 * args->workspace_bytes 0.  The workspace the call needs
 * (ssu_ssd_workspace_size) must fit SSU_SSD_STATIC_SCRATCH_BYTES (64 MiB: for
 * heads 128, dim 64, dstate 128 and chunk 256, up to 15 chunks);
 * a larger call returns SSU_ERR_INVALID before anything runs.  Nothing is
 * allocated: the scratch is a device array of the library, looked up once per
 * device on the first call made with that device current -- make that first
 * call before capturing a graph.  The scratch needs no initialisation.  Calls
 * that overlap in time (other streams, other threads) share the scratch and
 * corrupt each other's results: serialise them.  The 64 MiB are reserved on
 * every device that loads the library, for the life of the process, whether
 * or not this entry point is ever called.
 */
#define SSU_SSD_STATIC_SCRATCH_BYTES (64ull << 20)
ssu_status ssu_ssd_prefill_static(const ssu_ssd_args *args, void *stream);

/*
 * One copy of a batch: `bytes` bytes from device address `src` to device
 * address `dst` (any alignment; 16-byte aligned addresses take the vector
 * path).
 */
typedef struct ssu_copy {
    uint64_t src;
    uint64_t dst;
    uint64_t bytes;
} ssu_copy;

/*
 * Batched state copies with memmove semantics (digest of vLLM PR #50729,
 * section 实现拆解: speculative decoding moves and shifts slot state inside
 * one buffer, so a copy's source and destination may overlap).  Each copy
 * leaves in its destination the bytes its source held before the copy, also
 * when the two ranges overlap; copies that do not overlap themselves run at
 * full parallelism, and only the ones that do are moved in order (by one
 * CTA each).
 *   copies     device [n] descriptors, 8-byte aligned.
 *   max_bytes  an upper bound on every copy's `bytes`; it sizes the grid.  A
 *              copy longer than max_bytes sets SSU_DEV_BAD_COPY and is
 *              skipped.
 *   d_status   device int32 or NULL (SSU_DEV_* bits ORed in).
 * Different copies of one call must not overlap one another (no copy reads
 * or writes bytes another copy writes); the result would depend on
 * scheduling.  Copies with bytes == 0 or src == dst do nothing.  n == 0 or
 * max_bytes == 0 launches nothing.  No article on the pages gives this an
 * API; the descriptor form is this library's.
 */
ssu_status ssu_batch_copy(const ssu_copy *copies, int64_t n, uint64_t max_bytes, int32_t *d_status,
                          void *stream);

/*
 * The read copy (see ssu_replay_buffers) of `rows` consecutive state rows of
 * `dstate` elements: state rows r in [0, rows) of `state` (state_dtype) into
 * `shadow` rows (format SSU_SHADOW_F16, SSU_SHADOW_E4M3 or SSU_SHADOW_NVFP4)
 * and, for E4M3, `scale[r]`, for NVFP4 the record of SSU_NVFP4_SCALE_WORDS
 * floats at scale + r * SSU_NVFP4_SCALE_WORDS(dstate) (dstate a multiple of
 * 32; the record's padding is left as it is).  Use it to build the copy of
 * checkpoints written by other means (a prefill, a copy).  rows == 0 launches
 * nothing.
 */
ssu_status ssu_shadow_refresh(const void *state, int32_t state_dtype, int64_t rows, int64_t dstate,
                              int32_t format, void *shadow, float *scale, void *stream);

/*
 * Get the kernel for one configuration ready before any CUDA graph capture:
 * checks that the configuration is supported, loads the kernel's module on
 * the current device and caches its launch attributes.  MATE "Mamba / SSU",
 * Graph capture and prewarm_selective_state_update (kernels there are
 * compiled at first use; here they are compiled ahead of time, so this only
 * loads them).  `packed` selects the packed kernel instead of the one-token
 * kernel.  Returns SSU_ERR_UNSUPPORTED for a dstate or dtype the kernels do
 * not cover.
 */
ssu_status ssu_prewarm(int32_t state_dtype, int32_t io_dtype, int32_t dt_dtype,
                       int64_t heads, int64_t dim, int64_t dstate, int64_t groups,
                       int32_t packed);

/*
 * Self-test of the kernels' exit path, for tests only: ssu_update_onetoken
 * with every bounded wait limited to `wait_cycles` SM clock cycles (1000 up
 * to the default of about a second) and the stage of unit `withhold_unit`
 * (units are numbered (b * heads + h) * dim_tiles + dim_tile, dim tiles of
 * 64 rows) never filled.  The consumers' wait for that unit runs out with no
 * copy pending; the CTA that owns the unit stops issuing copies, waits for
 * the copies it already issued, sets SSU_DEV_TIMEOUT in *d_status and
 * returns.  The results of that CTA's remaining units are left unwritten;
 * every other CTA completes normally.  No device fault is involved and the
 * context stays usable.
 */
ssu_status ssu_selftest_timeout(const ssu_args *args, int64_t batch, const ssu_slot_table *read,
                                const ssu_slot_table *dst, int64_t withhold_unit, int64_t wait_cycles,
                                void *stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char *ssu_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SSU_H */
