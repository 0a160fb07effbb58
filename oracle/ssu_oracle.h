/*
 * ssu_oracle.h -- interface of the double-precision CPU oracle for the
 * Mamba-2 selective state update.  TEST INFRASTRUCTURE ONLY: used by the
 * tests, the smoke check and the CPU-baseline leg of the benchmark, never by
 * the library under test.  Host pointers only; every array is contiguous.
 */
#ifndef SSU_ORACLE_H
#define SSU_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element formats (raw bits in host memory) */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_F64 = 3 };
/* return codes */
enum { ORC_OK = 0, ORC_INVALID = 1, ORC_ALIASING = 2 };
/* slot-table addressing */
enum { ORC_SLOTS_STRIDED = 0, ORC_SLOTS_PER_ROW = 1 };
/* bits of slot_touched[] */
enum { ORC_TOUCH_READ = 1, ORC_TOUCH_WRITTEN = 2 };

typedef struct {
    const int64_t *entries;  /* NULL: no table                             */
    int64_t s0, s1;          /* STRIDED: entry = b*s0 + step*s1            */
    int64_t extent;          /* entries[0 .. extent-1] are addressable     */
    int32_t mode;            /* ORC_SLOTS_STRIDED or ORC_SLOTS_PER_ROW     */
} orc_table;

typedef struct {
    int64_t slots, heads, dim, dstate, groups;
    int32_t state_dtype, io_dtype, dt_dtype;
    int32_t dt_per_head;            /* dt is [rows, heads] instead of [rows, heads, dim] */
    const void *state_in;           /* [slots, heads, dim, dstate], read only              */
    void *state_out;                /* same shape; caller fills it with state_in first     */
    const void *x, *dt, *B, *C, *z; /* x, z: [rows, heads, dim]; B, C: [rows, groups, dstate]; z may be NULL */
    const float *A, *D, *dt_bias;   /* [heads] fp32; D and dt_bias may be NULL             */
    void *y;                        /* [rows, heads, dim] in io_dtype, rounded to nearest even */
    double *y_exact;                /* [rows, heads, dim] before rounding; may be NULL     */
    int32_t dt_softplus, disable_state_update;
    int64_t pad_slot_id;
    int64_t nseq, rows;
    const int64_t *cu_seqlens;      /* [nseq + 1]; NULL: sequence b is row b (one token)  */
    const int64_t *num_accepted;    /* [nseq]; NULL: seed at step 0                       */
    orc_table read, dst;            /* dst.entries NULL: publish through the read table   */
    uint8_t *slot_touched;          /* [slots] or NULL: OR of ORC_TOUCH_* per slot         */
} orc_problem;

int orc_ssu_run(const orc_problem *problem, char *err, int errlen);

/* One decode token per sequence with the state kept as a checkpoint plus a
 * buffer of the inputs of the steps since the last fold (article "ReplaySSM:
 * Cache SSM Inputs, Not State", section 核心做法).  All arrays contiguous. */
typedef struct {
    int64_t slots, heads, dim, dstate, groups;
    int32_t state_dtype, io_dtype, dt_dtype;
    int32_t dt_per_head;
    const void *ckpt_in;            /* [slots, heads, dim, dstate] checkpoints, read only        */
    void *ckpt_out;                 /* same shape; caller fills it with ckpt_in first            */
    const void *x, *dt, *B, *C, *z; /* current token: x, z [batch, heads, dim]; B, C [batch, groups, dstate] */
    const float *A, *D, *dt_bias;
    void *y;                        /* [batch, heads, dim] io dtype                               */
    double *y_exact;                /* [batch, heads, dim] or NULL                                */
    int32_t dt_softplus;
    int64_t pad_slot_id;
    int64_t batch;
    const int64_t *slot_of;         /* [batch] slot of each sequence; NULL: slot b                */
    int64_t len;                    /* buffer length L >= 1                                       */
    void *xbuf;                     /* [slots, L, heads, dim] io dtype, in/out                    */
    float *dtbuf;                   /* [slots, L, heads, dim] fp32 processed steps, in/out         */
    void *Bbuf;                     /* [slots, L, groups, dstate] io dtype, in/out                */
    const int64_t *count_in;        /* [batch] entries buffered before the call (0 <= c < L)      */
    int64_t *count_out;             /* [batch] entries buffered after the call                    */
    int32_t shadow_format;          /* ORC_SHADOW_*: the low-precision read copy, or none         */
    void *shadow;                   /* [slots, heads, dim, dstate] codes, in/out (NULL: none)     */
    float *shadow_scale;            /* [slots, heads, dim] row scales (E4M3) or scale records
                                       (NVFP4), in/out                                             */
} orc_replay_problem;

/* Packed variable-length SSD prefill (MATE documentation, page "Mamba / SSU",
 * "SSD packed prefill" and the API reference of ssd_combined_fwd_varlen).
 * What it computes is the Mamba-2 recurrence over each sequence's tokens
 * (the chunked five-stage evaluation is a reordering of it): for token t of
 * head h, dim row p, g = h / (heads / groups),
 *     dt' = clamp(softplus?(dt[t,h] + dt_bias[h]), dt_lo, dt_hi)
 *     S[n] = S[n] exp(A[h] dt') + dt' x[t,h,p] B[t,g,n]
 *     y[t,h,p] = (sum_n S[n] C[t,g,n] + D[h] x[t,h,p]) * silu(z[t,h,p])
 * Chunk c covers tokens [cu_chunk[c], cu_chunk[c+1]); chunks are visited in
 * order; a chunk opens a sequence when c == 0 or seq_idx[c] != seq_idx[c-1],
 * and its entering state is then initial_states[seq_idx[c]] (zero without
 * initial states); otherwise it is the state the previous chunk left.  The
 * state is carried in double; states[c] = the state at the end of chunk c,
 * rounded to state_dtype.  All arrays contiguous. */
typedef struct {
    int64_t tokens, heads, dim, dstate, groups, nchunks, nseq;
    int32_t io_dtype, dt_dtype, state_dtype;
    const void *x, *dt, *B, *C, *z;   /* x, z [tokens, heads, dim]; dt [tokens, heads]; B, C [tokens, groups, dstate] */
    const float *A, *D, *dt_bias;     /* [heads]; D, dt_bias may be NULL                               */
    int32_t dt_softplus;
    double dt_lo, dt_hi;              /* dt_limit                                                      */
    const int64_t *cu_chunk;          /* [nchunks + 1]                                                 */
    const int64_t *seq_idx;           /* [nchunks], each in [0, nseq)                                  */
    const void *initial_states;       /* [nseq, heads, dim, dstate] in state_dtype, or NULL            */
    void *y;                          /* [tokens, heads, dim] io_dtype                                 */
    double *y_exact;                  /* [tokens, heads, dim] or NULL                                  */
    void *states;                     /* [nchunks, heads, dim, dstate] state_dtype                      */
} orc_ssd_problem;

int orc_ssd_run(const orc_ssd_problem *problem, char *err, int errlen);

/* Low-precision read copy of the checkpoints (article "ReplaySSM", section
 * 低精度读写分离): steps that do not fold read it instead of the checkpoint;
 * a fold rewrites it from the new checkpoint.
 *   ORC_SHADOW_F16   binary16, round to nearest even.
 *   ORC_SHADOW_E4M3  OCP FP8 E4M3 (bias 7, 3 fraction bits, no infinities,
 *                    largest 448) with one fp32 scale per state row: amax =
 *                    the row's largest magnitude, code = E4M3(v * 448 / amax)
 *                    with the quotient in double, rounded to nearest even;
 *                    scale = amax / 448 stored in fp32 (1, and zero codes,
 *                    for an all-zero row); value = E4M3 value * scale.
 *   ORC_SHADOW_NVFP4 FP4 E2M1 codes (two a byte, the even element in the low
 *                    nibble) with two scale levels: per row the fp32 scale
 *                    s = amax / (6 * 448); per block of 16 elements the E4M3
 *                    code of (block amax) / (6 s); code = E2M1(v / (block
 *                    scale * s)), quotients in double, roundings to nearest
 *                    even, saturating.  `scale` holds one record per row of
 *                    orc_nvfp4_scale_words(dstate) floats: s, then the block
 *                    scale codes as bytes.  value = E2M1 * block scale * s.
 *                    dstate a multiple of 16. */
enum { ORC_SHADOW_NONE = 0, ORC_SHADOW_F16 = 1, ORC_SHADOW_E4M3 = 2, ORC_SHADOW_NVFP4 = 3 };

/* The read copy of `rows` state rows of `dstate` elements (`state` in
 * state_dtype); `scale` may be NULL for ORC_SHADOW_F16. */
int orc_shadow_refresh(const void *state, int32_t state_dtype, int64_t rows, int64_t dstate, int32_t format,
                       void *shadow, float *scale);
uint8_t orc_e4m3_encode(double v);
double orc_e4m3_decode(uint8_t code);
uint8_t orc_e2m1_encode(double v);
double orc_e2m1_decode(uint8_t code);
int64_t orc_nvfp4_scale_words(int64_t dstate);

int orc_replay_run(const orc_replay_problem *problem, char *err, int errlen);

/* Speculative decoding on the checkpoint + buffer form (article "ReplaySSM:
 * Cache SSM Inputs, Not State", section 投机解码回滚).  Each sequence brings
 * T draft tokens: x, z [batch, T, heads, dim]; dt [batch, T, heads, dim] (or
 * [batch, T, heads] with dt_per_head); B, C [batch, T, groups, dstate]; y
 * [batch, T, heads, dim].  With c = count_in[b] committed entries:
 *   - if c + 2T >= L the c entries are first folded into the checkpoint
 *     (written back once, in state_dtype) and c becomes 0 -- the flush one
 *     window early, so that the next step always has T free entries;
 *   - the drafts are appended as entries c .. c+T-1 (x and B keep their bits,
 *     the processed step is stored in fp32);
 *   - draft k's output is read from the state after entries 0 .. c+k, i.e.
 *     the checkpoint as stored, the committed entries and drafts 0 .. k in
 *     order (causal mask), with every step's dt' as stored in fp32;
 *   - count_out[b] = c: nothing is committed; the caller advances the count
 *     by the accepted prefix, and later entries are simply overwritten.
 * A pad slot has no history and no checkpoint: zero state, the drafts only,
 * nothing written, count 0.  The other fields mean what they mean for
 * orc_replay_run (no read copy). */
typedef struct {
    int64_t slots, heads, dim, dstate, groups;
    int32_t state_dtype, io_dtype, dt_dtype;
    int32_t dt_per_head;
    const void *ckpt_in;            /* [slots, heads, dim, dstate] checkpoints, read only        */
    void *ckpt_out;                 /* same shape; caller fills it with ckpt_in first            */
    const void *x, *dt, *B, *C, *z; /* the drafts, see above                                     */
    const float *A, *D, *dt_bias;
    void *y;                        /* [batch, T, heads, dim] io dtype                            */
    double *y_exact;                /* [batch, T, heads, dim] or NULL                             */
    int32_t dt_softplus;
    int64_t pad_slot_id;
    int64_t batch, ntok;            /* sequences, drafts per sequence (T >= 1, T <= L)            */
    const int64_t *slot_of;         /* [batch] slot of each sequence; NULL: slot b                */
    int64_t len;                    /* buffer length L                                            */
    void *xbuf;                     /* [slots, L, heads, dim] io dtype, in/out                    */
    float *dtbuf;                   /* [slots, L, heads, dim] fp32 processed steps, in/out         */
    void *Bbuf;                     /* [slots, L, groups, dstate] io dtype, in/out                */
    const int64_t *count_in;        /* [batch] committed entries (0 <= c < L)                     */
    int64_t *count_out;             /* [batch] committed entries after the call                   */
} orc_verify_problem;

int orc_replay_verify_run(const orc_verify_problem *problem, char *err, int errlen);

double orc_softplus(double v);
double orc_silu(double z);
double orc_decode(uint32_t bits, int dtype);
uint32_t orc_encode(double v, int dtype);

#ifdef __cplusplus
}
#endif

#endif /* SSU_ORACLE_H */
