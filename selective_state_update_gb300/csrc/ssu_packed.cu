// ssu_packed.cu -- packed variable-length and multi-token (MTP) decode.
// Calls whose sequences are long (kLongRowsPerSeq tokens or more on average,
// known on the host from rows / nseq) go to ssu_packed_long.cu instead.
//
// MATE documentation, page "Mamba / SSU", "SSU at a glance", rows Sequence
// layout, Slot semantics and Variable-length and MTP decode: cu_seqlens splits
// the packed rows between sequences; the read slot is seeded at
// max(num_accepted - 1, 0); every token publishes its state to its own
// destination entry (or its own read-table entry without a destination
// table); pad destinations are never written; empty sequences are skipped.
// Section Graph capture: one launch, no host/device scalar copies.
//
// Work unit: (sequence b, head h, tile of kTileRows dim rows).  The kernel is
// persistent and warp-specialised, like the one-token kernel:
//   work split  each CTA takes one contiguous run of units, cut so that every
//               CTA gets the same share of the call's weight, a unit weighing
//               its sequence's length plus one (the seed read).  Sequence
//               lengths live on the device, so the producer finds its run's
//               first unit by a 32-way search over cu_seqlens; the tail is at
//               most one unit.  Consecutive units of a run are the heads of
//               one sequence, so a sequence's rows, seed slot and
//               destinations are resolved once for all its heads.
//   producer    one warp, pure data movement, up to kStages ring stages ahead:
//               per stage (a unit's chunk of up to kTokChunk tokens) it writes
//               the header (destination slot of each token, packed row, head
//               scalars) and starts bulk asynchronous copies (TMA engine) of
//               the seed tile (first chunk only) and of every token's B, C,
//               x, z and dt rows, all completing on the stage's "full"
//               mbarrier; operands whose rows are not 16-byte aligned are
//               copied by the warp's lanes instead.
//   consumers   carry the unit's fp32 state in registers (kPackedRows rows x
//               16 values per thread) across all its tokens and chunks.  Per
//               stage they first turn the staged inputs of every (token, row)
//               into its row scalars {dA, dt' x, x, gate}, one thread each, so
//               that the transcendental work runs in parallel rather than on
//               each token's critical path; then per token they update the
//               rows, write y and publish the rounded state to the token's
//               destination slot with 16-byte streaming stores; the stage is
//               released as soon as its chunk is done.
// The state is read from HBM once per unit and written once per token; the
// seed reads of the next units are in flight while the consumers compute.
#include <atomic>

#include "ssu_device.cuh"

namespace ssu {

namespace {

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Tokens staged per ring stage; longer sequences take several stages.  Eight
// measured faster than four (a deeper ring of smaller stages) on short
// sequences: the per-stage work of the consumers weighs more than the ring
// depth.
constexpr int kTokChunk = 8;
// State rows per consumer thread: two (kPackedSlots = 32 row slots of L
// lanes), so that a CTA has eight consumer warps at dstate 128 to hide the
// latency of each token's dependent steps.
constexpr int kPackedRows = 2;
constexpr int kPackedSlots = kTileRows / kPackedRows;

struct PackedHeader {
    int64_t ws[kTokChunk];  // destination slot of each token, -1: not written
    int64_t r0;             // packed row of the chunk's first token
    int32_t flags;          // kChunk* bits
    int32_t ntok;           // tokens in this chunk
    int32_t h, row0, rows_here;
    float Ah, bias, Dh;
};
enum : int32_t { kChunkFirst = 1, kChunkSeeded = 2, kChunkStop = 4 };

template <typename TS, int L>
struct PackedPipe {
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kSeedBytes = kTileRows * kN * static_cast<int>(sizeof(TS));
    // One token's operands as stored (B, C: dstate values; x, z, dt: the
    // tile's rows), each part 16-byte aligned, and for 16-bit B and C their
    // fp32 values: at most 2 N 4 + 3 kTileRows 4 bytes (4-byte io) or
    // 2 N 2 + 2 kTileRows 2 + kTileRows 4 + 2 N 4 (16-bit io).
    static constexpr int kOpBytes4 = 2 * kN * 4 + 3 * kTileRows * 4;
    static constexpr int kOpBytes2 = 2 * kN * 2 + 2 * kTileRows * 2 + kTileRows * 4 + 2 * kN * 4;
    static constexpr int kOpBytesMax = kOpBytes4 > kOpBytes2 ? kOpBytes4 : kOpBytes2;
    // the row scalars of every (token, row) of the chunk, float4 each
    static constexpr int kRowqOffset = kSeedBytes + kTokChunk * kOpBytesMax;
    static constexpr int kHeaderOffset = kRowqOffset + kTokChunk * kTileRows * 16;
    static constexpr int kStageBytes = align_up(kHeaderOffset + static_cast<int>(sizeof(PackedHeader)), 128);
    static constexpr int kConsumerThreads = kPackedSlots * L;
    static constexpr int kConsumerWarps = (kConsumerThreads + 31) / 32;
    static constexpr int kConsumers = 32 * kConsumerWarps;
    static constexpr int kThreads = 32 * (kConsumerWarps + 1);
    // Dynamic shared memory of an SM (228 KB, 1 KB of it reserved per CTA):
    // two CTAs when each still gets a ring of two stages or more and the
    // register file holds a thread's 32 state values plus B and C at two
    // CTAs (up to nine warps a CTA), else one CTA with the deeper ring.
    static constexpr int kSmemPerSm = 228 * 1024;
    static constexpr int kCtasPerSm =
        (kThreads <= 288 && (kSmemPerSm / 2 - 1024 - 256) / kStageBytes >= 2) ? 2 : 1;
    static constexpr int kFit = (kSmemPerSm / kCtasPerSm - 1024 - 256) / kStageBytes;
    static constexpr int kStages = kFit < 6 ? kFit : 6;
    static constexpr int kBarOffset = kStages * kStageBytes;
    static constexpr int kExitOffset = kBarOffset + 2 * kStages * 8;
    static constexpr int kBytes = kExitOffset + static_cast<int>(sizeof(RingExit));
    static_assert(kStages >= 2 && kStages <= kMaxRingStages, "ring of two to eight stages");
    static_assert(kBytes <= 227 * 1024, "stage ring larger than a CTA's shared memory");
};

// Byte offsets of a token's operands within its slot of the stage: B, C, x,
// z, dt as stored, then (16-bit io) B and C as fp32.  offBf / offCf give the
// fp32 B and C either way.
struct OpLayout {
    int io, dts, offC, offX, offZ, offDT, offBf, offCf, stride;
    __device__ __forceinline__ OpLayout(const KParams &p) {
        io = p.io_dtype == kF32 ? 4 : 2;
        dts = p.dt_dtype == kF32 ? 4 : 2;
        offC = align_up(p.N * io, 16);
        offX = offC + align_up(p.N * io, 16);
        offZ = offX + align_up(kTileRows * io, 16);
        offDT = offZ + align_up(kTileRows * io, 16);
        const int end = offDT + align_up(kTileRows * dts, 16);
        if (io == 4) {
            offBf = 0;
            offCf = offC;
            stride = end;
        } else {
            offBf = end;
            offCf = end + p.N * 4;
            stride = end + 2 * p.N * 4;
        }
    }
};

// The sequence a producer is walking, resolved once for all of its heads.
struct SeqInfo {
    int64_t b, start, len, rs;
    int64_t span;     // cu_seqlens[b + 1] - cu_seqlens[b] as given (the work split's weight)
    int64_t ws_lane;  // destination slot of token `lane` (< 32), -1: not written
    bool ok;          // rows, seed and every destination valid, len > 0
};

__device__ __forceinline__ int64_t seq_start(const KParams &p, int64_t b) {
    return p.cu != nullptr ? load_index(p.cu, b, p.meta_is_i64) : b * p.steps;
}

// Destination slot of token t of sequence b (-1: not written); false if the
// entry or slot is invalid (flagged).
__device__ __forceinline__ bool dst_slot(const KParams &p, const SlotTab &wt, int64_t b, int64_t t, int64_t start,
                                         int64_t *ws) {
    int64_t w;
    if (!table_slot(p, wt, b, t, start, b, &w) || !slot_ok(p, w)) return false;
    *ws = (p.disable || w == p.pad) ? -1 : w;
    return true;
}

// Everything about sequence b the producer needs (all lanes get the same
// result; lane t also keeps the destination of token t).
__device__ SeqInfo load_seq(const KParams &p, int64_t b, int lane) {
    SeqInfo q;
    q.b = b;
    q.ok = false;
    q.len = 0;
    q.rs = 0;
    q.ws_lane = -1;
    const int64_t start = seq_start(p, b);
    const int64_t end = p.cu != nullptr ? load_index(p.cu, b + 1, p.meta_is_i64) : start + p.steps;
    q.start = start;
    q.span = end - start;
    if (start < 0 || end < start || end > p.rows) {
        if (lane == 0) flag(p.status, kDevBadSeqlen);
        return q;
    }
    q.len = end - start;
    if (q.len == 0) return q;
    int64_t t_seed = 0;
    if (p.acc != nullptr) {
        t_seed = load_index(p.acc, b, p.meta_is_i64) - 1;
        if (t_seed < 0) t_seed = 0;
    }
    // Per-row tables hold one entry per packed row: the seed step must be
    // one of the sequence's own rows.
    if (p.rd.entries != nullptr && p.rd.per_row && t_seed >= q.len) {
        if (lane == 0) flag(p.status, kDevBadEntry);
        return q;
    }
    int bad = 0;
    if (lane == 0) {
        int64_t rs;
        if (table_slot(p, p.rd, b, t_seed, start, b, &rs) && slot_ok(p, rs))
            q.rs = rs;
        else
            bad = 1;
    }
    q.rs = __shfl_sync(0xffffffffu, q.rs, 0);
    // Every destination of the sequence is checked before anything is written.
    const SlotTab &wt = (p.wr.entries != nullptr) ? p.wr : p.rd;
    for (int64_t t = lane; t < q.len; t += 32) {
        int64_t ws;
        if (!dst_slot(p, wt, b, t, start, &ws))
            bad = 1;
        else if (t < 32)
            q.ws_lane = ws;
    }
    q.ok = !__any_sync(0xffffffffu, bad);
    return q;
}

// Whether cu_seqlens starts at or above 0, ends at or below the row count and
// never decreases in between (each lane checks every 32nd step; the whole
// warp gets the answer).
__device__ bool cu_monotone(const KParams &p, int lane) {
    bool ok = lane != 0 || (load_index(p.cu, 0, p.meta_is_i64) >= 0 &&
                            load_index(p.cu, p.nseq, p.meta_is_i64) <= p.rows);
    for (int64_t b = lane; b < p.nseq; b += 32)
        ok &= load_index(p.cu, b + 1, p.meta_is_i64) >= load_index(p.cu, b, p.meta_is_i64);
    return __all_sync(0xffffffffu, ok);
}

// The work split.  Units are numbered u = (b * H + h) * ptiles + pt.  With a
// non-decreasing cu_seqlens a unit of sequence b weighs len_b + 1 and the
// weight before sequence b is HP * (cu[b] - cu[0] + b), HP = H * ptiles (the
// dense form: len_b = steps); otherwise every unit weighs 1.  Every CTA
// computes the same weights, so the runs [lo, hi) of the CTAs cover every
// unit exactly once.
struct Split {
    bool weighted;
    int64_t cu0, HP;
    __device__ __forceinline__ int64_t before(const KParams &p, int64_t b) const {
        if (p.cu == nullptr) return HP * b * (p.steps + 1);
        return weighted ? HP * (load_index(p.cu, b, p.meta_is_i64) - cu0 + b) : HP * b;
    }
    __device__ __forceinline__ int64_t unit_weight(const SeqInfo &q) const {
        return weighted ? q.span + 1 : 1;
    }
    // The largest b < nseq whose prefix weight is <= target: a 32-way search
    // by the warp (the prefix never decreases, so the lanes below the cut
    // form a prefix of the warp).
    __device__ int64_t find(const KParams &p, int64_t target, int lane) const {
        if (p.cu == nullptr || !weighted) {
            const int64_t b = target / (p.cu == nullptr ? HP * (p.steps + 1) : HP);
            return b < p.nseq - 1 ? b : p.nseq - 1;
        }
        int64_t lo = 0, hi = p.nseq;
        while (hi - lo > 1) {
            const int64_t stride = (hi - lo + 31) / 32;
            const int64_t m = lo + lane * stride;
            const bool le = m < hi && before(p, m) <= target;
            const unsigned ball = __ballot_sync(0xffffffffu, le);
            const int last = 31 - __clz(ball);
            lo += last * stride;
            hi = lo + stride < hi ? lo + stride : hi;
        }
        return lo;
    }
};

template <typename TS, int L>
__device__ __forceinline__ unsigned char *stage_base(unsigned char *smem, int s) {
    return smem + s * PackedPipe<TS, L>::kStageBytes;
}

// `count` elements of `bytes` each from a row of a small operand (element
// stride `stride`) into shared memory: one bulk copy when `bulk`, else by the
// warp's lanes (stride 0 replicates one element).  Returns the bytes the bulk
// copy will complete on `bar` (0 for lane copies).
__device__ __forceinline__ uint32_t stage_row(unsigned char *dst, const void *base, int64_t off, int64_t stride,
                                              int count, int bytes, bool bulk, uint64_t *bar, int lane, int who) {
    if (bulk) {
        const uint32_t n = static_cast<uint32_t>(count * bytes);
        if (lane == who) bulk_load(dst, static_cast<const unsigned char *>(base) + off * bytes, n, bar);
        return n;
    }
    for (int i = lane; i < count; i += 32) {
        if (bytes == 4)
            reinterpret_cast<uint32_t *>(dst)[i] = __ldg(static_cast<const unsigned int *>(base) + off + i * stride);
        else
            reinterpret_cast<unsigned short *>(dst)[i] =
                __ldg(static_cast<const unsigned short *>(base) + off + i * stride);
    }
    return 0;
}

// Fill stage k with chunk [t0, t0 + ntok) of unit (q.b, h, pt).  Returns false
// when the CTA stops (a wait gave up or another role aborted).
template <typename TS, int L>
__device__ bool fill_chunk(const KParams &p, const SeqInfo &q, int h, int pt, int64_t t0, int ntok, float Ah,
                           float bias, float Dh, int k, unsigned char *smem, uint64_t *full, uint64_t *empty,
                           RingExit *rx, const OpLayout &ol, int lane) {
    using PS = PackedPipe<TS, L>;
    constexpr int S = PS::kStages;
    constexpr int N = PS::kN;
    const int s = k % S, round = k / S;
    if (ring_aborted(rx)) return false;
    if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1, p.wait_cycles)) {
        if (lane == 0) {
            flag(p.status, kDevTimeout);
            ring_abort(rx);
        }
        return false;
    }
    unsigned char *st = stage_base<TS, L>(smem, s);
    PackedHeader *hd = reinterpret_cast<PackedHeader *>(st + PS::kHeaderOffset);
    const int row0 = pt * kTileRows;
    const int rows_here = min(kTileRows, p.P - row0);
    const bool first = t0 == 0;
    const bool seeded = first && q.rs != p.pad;
    // Destinations of the chunk's tokens: token t0 + i goes to header entry
    // i; lane t holds token t's slot for t < 32 (t0 is a multiple of
    // kTokChunk, so t0 + i < 32 whenever t0 < 32).
    int64_t ws = -1;
    if (t0 < 32) {
        const int src = static_cast<int>(t0) + lane;
        ws = __shfl_sync(0xffffffffu, q.ws_lane, src < 32 ? src : 31);
    } else if (lane < ntok) {
        const SlotTab &wt = (p.wr.entries != nullptr) ? p.wr : p.rd;
        dst_slot(p, wt, q.b, t0 + lane, q.start, &ws);  // validated when the sequence was loaded
    }
    if (lane < ntok) hd->ws[lane] = ws;
    if (lane == 0) {
        hd->r0 = q.start + t0;
        hd->flags = (first ? kChunkFirst : 0) | (seeded ? kChunkSeeded : 0);
        hd->ntok = ntok;
        hd->h = h;
        hd->row0 = row0;
        hd->rows_here = rows_here;
        hd->Ah = Ah;
        hd->bias = bias;
        hd->Dh = Dh;
    }
    // Bytes the bulk copies will bring (the same on every lane).
    uint32_t tx = 0;
    if (seeded) tx += static_cast<uint32_t>(rows_here) * N * sizeof(TS);
    if (p.bulk_ops & kBulkBC) tx += 2u * ntok * N * ol.io;
    if (p.bulk_ops & kBulkXZ) tx += (p.z != nullptr ? 2u : 1u) * ntok * rows_here * ol.io;
    if (p.bulk_ops & kBulkDT) tx += static_cast<uint32_t>(ntok) * rows_here * ol.dts;
    if (lane == 0 && tx > 0) mbar_arrive_expect(&full[s], tx);
    __syncwarp();
    if (seeded && lane == 0) {
        const TS *src = static_cast<const TS *>(p.state) + ((q.rs * p.H + h) * static_cast<int64_t>(p.P) + row0) * N;
        bulk_load(st, src, static_cast<uint32_t>(rows_here) * N * sizeof(TS), &full[s]);
    }
    const int g = h / p.heads_per_group;
    unsigned char *ops = st + PS::kSeedBytes;
    for (int t = 0; t < ntok; ++t) {
        const int64_t r = q.start + t0 + t;
        unsigned char *o = ops + t * ol.stride;
        // lanes 1..5 issue the bulk copies of one token, so they go out together
        stage_row(o, p.B, r * p.Bs[0] + g * p.Bs[1], p.Bs[2], N, ol.io, p.bulk_ops & kBulkBC, &full[s], lane, 1);
        stage_row(o + ol.offC, p.C, r * p.Cs[0] + g * p.Cs[1], p.Cs[2], N, ol.io, p.bulk_ops & kBulkBC, &full[s],
                  lane, 2);
        stage_row(o + ol.offX, p.x, r * p.xs[0] + h * p.xs[1] + row0 * p.xs[2], p.xs[2], rows_here, ol.io,
                  p.bulk_ops & kBulkXZ, &full[s], lane, 3);
        if (p.z != nullptr)
            stage_row(o + ol.offZ, p.z, r * p.zs[0] + h * p.zs[1] + row0 * p.zs[2], p.zs[2], rows_here, ol.io,
                      p.bulk_ops & kBulkXZ, &full[s], lane, 4);
        stage_row(o + ol.offDT, p.dt, r * p.dts[0] + h * p.dts[1] + row0 * p.dts[2], p.dts[2], rows_here, ol.dts,
                  p.bulk_ops & kBulkDT, &full[s], lane, 5);
    }
    if (lane == 0) ring_note_fill(rx, s, round);
    if (lane != 0 || tx == 0) mbar_arrive(&full[s]);
    return true;
}

// The final stage: tells the consumers that the run is done.
template <typename TS, int L>
__device__ bool post_stop(const KParams &p, int k, unsigned char *smem, uint64_t *full, uint64_t *empty,
                          RingExit *rx, int lane) {
    using PS = PackedPipe<TS, L>;
    constexpr int S = PS::kStages;
    const int s = k % S, round = k / S;
    if (ring_aborted(rx)) return false;
    if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1, p.wait_cycles)) {
        if (lane == 0) {
            flag(p.status, kDevTimeout);
            ring_abort(rx);
        }
        return false;
    }
    PackedHeader *hd = reinterpret_cast<PackedHeader *>(stage_base<TS, L>(smem, s) + PS::kHeaderOffset);
    if (lane == 0) {
        hd->flags = kChunkStop;
        hd->ntok = 0;
        ring_note_fill(rx, s, round);
    }
    mbar_arrive(&full[s]);
    return true;
}

template <typename TS, int L>
__device__ void packed_producer(const KParams &p, unsigned char *smem, uint64_t *full, uint64_t *empty,
                                RingExit *rx) {
    const int lane = threadIdx.x & 31;
    const OpLayout ol(p);
    Split sp;
    sp.HP = static_cast<int64_t>(p.H) * p.ptiles;
    sp.cu0 = p.cu != nullptr ? load_index(p.cu, 0, p.meta_is_i64) : 0;
    sp.weighted = p.cu == nullptr || cu_monotone(p, lane);
    const int64_t total = sp.before(p, p.nseq);
    const int64_t lo_w = static_cast<int64_t>(blockIdx.x) * total / gridDim.x;
    const int64_t hi_w = (static_cast<int64_t>(blockIdx.x) + 1) * total / gridDim.x;
    // The run's first unit: the first whose start weight is >= lo_w.
    int64_t b = sp.find(p, lo_w, lane);
    SeqInfo q = load_seq(p, b, lane);
    int64_t wb = sp.before(p, b);  // weight before sequence b
    int64_t unit_w = sp.unit_weight(q);
    int64_t j = lo_w > wb ? (lo_w - wb + unit_w - 1) / unit_w : 0;
    int64_t w = wb + j * unit_w;  // start weight of unit (b, j)
    int k = 0;
    while (true) {
        if (j >= sp.HP) {  // the next sequence
            if (++b >= p.nseq) break;
            wb += sp.HP * unit_w;
            w = wb;
            j = 0;
            q = load_seq(p, b, lane);
            unit_w = sp.unit_weight(q);
            continue;
        }
        if (w >= hi_w) break;
        if (q.ok) {
            const int h = static_cast<int>(j / p.ptiles), pt = static_cast<int>(j % p.ptiles);
            const float Ah = __ldg(p.A + h);
            const float bias = p.dt_bias ? __ldg(p.dt_bias + h) : 0.f;
            const float Dh = p.D ? __ldg(p.D + h) : 0.f;
            for (int64_t t0 = 0; t0 < q.len; t0 += kTokChunk) {
                const int ntok = static_cast<int>(q.len - t0 < kTokChunk ? q.len - t0 : kTokChunk);
                if (!fill_chunk<TS, L>(p, q, h, pt, t0, ntok, Ah, bias, Dh, k, smem, full, empty, rx, ol, lane))
                    return;
                ++k;
            }
        }
        ++j;
        w += unit_w;
    }
    post_stop<TS, L>(p, k, smem, full, empty, rx, lane);
}

// Where a group of four fp32 values of a widened dstate vector sits, in
// float4 units: element e of the vector belongs to lane (e / kVec) % L as
// values 4 q .. 4 q + 3 of its chunk k = e / (kVec L) (q = (e % kVec) / 4), and
// lane l's group (k, q) is stored at (k kVec / 4 + q) L + l.  The lanes of a
// row then read consecutive 16-byte pieces (with kVec = 8 the natural order
// would put them 32 bytes apart: two-way bank conflicts).
template <int kVec, int L>
__device__ __forceinline__ int widened_group(int e) {
    const int cc = e / kVec, q = (e % kVec) / 4;
    return ((cc / L) * (kVec / 4) + q) * L + cc % L;
}

// This thread's 16 values of a widened dstate vector, in the element layout
// of Tile::gather.
template <typename TS, int L>
__device__ __forceinline__ void gather_widened(const float *v4, int lane, float *v) {
    constexpr int kVec = Tile<TS, L>::kVec;
#pragma unroll
    for (int k = 0; k < Tile<TS, L>::kChunks; ++k) {
#pragma unroll
        for (int q = 0; q < kVec / 4; ++q) {
            const float4 f = reinterpret_cast<const float4 *>(v4)[(k * (kVec / 4) + q) * L + lane];
            v[k * kVec + 4 * q + 0] = f.x;
            v[k * kVec + 4 * q + 1] = f.y;
            v[k * kVec + 4 * q + 2] = f.z;
            v[k * kVec + 4 * q + 3] = f.w;
        }
    }
}

// Eight 16-bit values (one 16-byte piece, lower address first) widened to
// fp32, bit for bit as bits_to_float does one value: values 0-3 to lo,
// 4-7 to hi.
__device__ __forceinline__ void widen8(uint4 u, bool bf, float4 *lo, float4 *hi) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (bf) {
            f[2 * k] = __uint_as_float(w[k] << 16);
            f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        } else {
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            f[2 * k] = v.x;
            f[2 * k + 1] = v.y;
        }
    }
    *lo = make_float4(f[0], f[1], f[2], f[3]);
    *hi = make_float4(f[4], f[5], f[6], f[7]);
}

// Everything a chunk's tokens share before the token loop, spread over the
// consumer threads: 16-bit B and C converted to fp32 once, a 16-byte piece
// per thread, in the order of widened_group, and the row scalars {dA, dt' x, x, gate} of every (token, row)
// into `rowq` ([kTokChunk][kTileRows]), from the same non-inlined function as
// the other kernels, hence the same bits.  The index splits divide by
// compile-time powers of two.
template <typename TS, int L, int N>
__device__ __forceinline__ void chunk_prep(const KParams &p, unsigned char *ops, const OpLayout &ol, int ntok,
                                           int rows_here, float Ah, float bias, float4 *rowq, int tid,
                                           int nthreads) {
    if (ol.io == 2) {
        constexpr int kPieces = N / 8;
        const bool bf = p.io_dtype == kBF16;
        for (int i = tid; i < ntok * kPieces; i += nthreads) {
            const int t = i / kPieces, c = i - t * kPieces;
            unsigned char *o = ops + t * ol.stride;
            constexpr int kVec = Tile<TS, L>::kVec;
            const int g0 = widened_group<kVec, L>(8 * c), g1 = widened_group<kVec, L>(8 * c + 4);
            float4 *b4 = reinterpret_cast<float4 *>(o + ol.offBf), *c4 = reinterpret_cast<float4 *>(o + ol.offCf);
            widen8(reinterpret_cast<const uint4 *>(o)[c], bf, b4 + g0, b4 + g1);
            widen8(reinterpret_cast<const uint4 *>(o + ol.offC)[c], bf, c4 + g0, c4 + g1);
        }
    }
    for (int i = tid; i < ntok * kTileRows; i += nthreads) {
        const int t = i / kTileRows, rr = i - t * kTileRows;
        if (rr >= rows_here) continue;
        const unsigned char *o = ops + t * ol.stride;
        const float xv = ol.io == 4 ? reinterpret_cast<const float *>(o + ol.offX)[rr]
                                    : bits_to_float(reinterpret_cast<const unsigned short *>(o + ol.offX)[rr],
                                                    p.io_dtype);
        const float zv = p.z == nullptr ? 0.f
                         : ol.io == 4  ? reinterpret_cast<const float *>(o + ol.offZ)[rr]
                                       : bits_to_float(reinterpret_cast<const unsigned short *>(o + ol.offZ)[rr],
                                                       p.io_dtype);
        const float dv = ol.dts == 4 ? reinterpret_cast<const float *>(o + ol.offDT)[rr]
                                     : bits_to_float(reinterpret_cast<const unsigned short *>(o + ol.offDT)[rr],
                                                     p.dt_dtype);
        rowq[t * kTileRows + rr] = row_scalars(RowInputs{dv, xv, zv}, Ah, bias, p.softplus, p.z != nullptr);
    }
}

// Returns the ring index of the first stage not consumed.
template <typename TS, int L>
__device__ int packed_consumer(const KParams &p, unsigned char *smem, uint64_t *full, uint64_t *empty,
                               RingExit *rx) {
    using T = Tile<TS, L>;
    using PS = PackedPipe<TS, L>;
    constexpr int N = PS::kN;
    constexpr int S = PS::kStages;
    const int tid = threadIdx.x;
    const int lane = tid % L;
    const int slot_row = tid / L;
    // dstate 16 leaves half of the one consumer warp without rows: those
    // lanes only take part in the shuffles
    const bool active = tid < PS::kConsumerThreads;
    const OpLayout ol(p);
    float st[kPackedRows][kElemsPerThread];
    int k = 0;
    for (;; ++k) {
        const int s = k % S;
        const bool ok = mbar_wait_bounded(&full[s], (k / S) & 1, p.wait_cycles);
        unsigned char *stg = stage_base<TS, L>(smem, s);
        const PackedHeader *hd = reinterpret_cast<const PackedHeader *>(stg + PS::kHeaderOffset);
        const int flags = ok ? hd->flags : kChunkStop;  // the header is read only from a full stage
        float4 *rowq = reinterpret_cast<float4 *>(stg + PS::kRowqOffset);
        if (!(flags & kChunkStop))
            chunk_prep<TS, L, N>(p, stg + PS::kSeedBytes, ol, hd->ntok, hd->rows_here, hd->Ah, hd->bias, rowq, tid,
                          PS::kConsumers);
        // The chunk's one barrier: its row scalars are ready, and every
        // consumer learns whether any wait gave up, so that all stop together
        // rather than leave the others at a barrier.
        if (barrier_or(1, PS::kConsumers, !ok)) {
            if (tid == 0) {
                flag(p.status, kDevTimeout);
                ring_abort(rx);
            }
            break;
        }
        if (flags & kChunkStop) {
            ++k;
            break;
        }
        const int ntok = hd->ntok, h = hd->h, row0 = hd->row0, rows_here = hd->rows_here;
        const int rows_mine = active ? rows_here : 0;
        const float Dh = hd->Dh;
        const int64_t r0 = hd->r0;
        if (flags & kChunkFirst) {
            const TS *seed = reinterpret_cast<const TS *>(stg);
#pragma unroll
            for (int j = 0; j < kPackedRows; ++j) {
                const int rr = slot_row + j * kPackedSlots;
                if ((flags & kChunkSeeded) && rr < rows_mine) {
                    T::load_row_smem(seed + rr * N, lane, st[j]);
                } else {
#pragma unroll
                    for (int i = 0; i < kElemsPerThread; ++i) st[j][i] = 0.f;
                }
            }
        }
        // offsets that stay fixed over the chunk's tokens
        const int64_t head_rows = (static_cast<int64_t>(h) * p.P + row0) * N;
        int64_t yo[kPackedRows];
        int rq[kPackedRows];
#pragma unroll
        for (int j = 0; j < kPackedRows; ++j) {
            const int rr = slot_row + j * kPackedSlots;
            rq[j] = rr < rows_mine ? rr : -1;
            yo[j] = r0 * p.ys[0] + h * p.ys[1] + (row0 + rr) * p.ys[2];
        }
        const int64_t slot_elems = static_cast<int64_t>(p.H) * p.P * N;
        for (int t = 0; t < ntok; ++t) {
            const unsigned char *o = stg + PS::kSeedBytes + t * ol.stride;
            float bv[kElemsPerThread], cv[kElemsPerThread];
            if (ol.io == 4) {  // as staged
                T::gather(reinterpret_cast<const float *>(o + ol.offBf), lane, bv);
                T::gather(reinterpret_cast<const float *>(o + ol.offCf), lane, cv);
            } else {  // as widened
                gather_widened<TS, L>(reinterpret_cast<const float *>(o + ol.offBf), lane, bv);
                gather_widened<TS, L>(reinterpret_cast<const float *>(o + ol.offCf), lane, cv);
            }
            const int64_t ws = hd->ws[t];
            TS *dst = ws >= 0 ? static_cast<TS *>(p.state) + ws * slot_elems + head_rows : nullptr;
#pragma unroll
            for (int j = 0; j < kPackedRows; ++j) {
                const float4 q = rowq[t * kTileRows + (rq[j] >= 0 ? rq[j] : 0)];
                const float sum = row_sum<L>(update_elems(st[j], bv, cv, q.x, q.y));
                if (rq[j] >= 0) {
                    if (lane == 0) store_small(p.y, yo[j] + t * p.ys[0], p.io_dtype, output(sum, Dh, q.z, q.w));
                    if (dst != nullptr) T::store_row(dst + rq[j] * N, lane, st[j]);
                }
            }
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&empty[s]);
    }
    return k;
}

// CTAs per SM from the ring's shared memory; the register budget follows.
template <typename TS, int L>
__global__ void __launch_bounds__(PackedPipe<TS, L>::kThreads, PackedPipe<TS, L>::kCtasPerSm)
    ssu_packed_kernel(const KParams p) {
    using PS = PackedPipe<TS, L>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + PS::kBarOffset);
    uint64_t *empty = full + PS::kStages;
    RingExit *rx = reinterpret_cast<RingExit *>(smem + PS::kExitOffset);
    if (threadIdx.x == 0) {
        for (int s = 0; s < PS::kStages; ++s) {
            mbar_init(&full[s], 32);
            mbar_init(&empty[s], PS::kConsumerWarps);
        }
        ring_init(rx);
    }
    __syncthreads();
    const int warp = threadIdx.x / 32;
    int consumed = 0;
    if (warp == PS::kConsumerWarps)
        packed_producer<TS, L>(p, smem, full, empty, rx);
    else
        consumed = packed_consumer<TS, L>(p, smem, full, empty, rx);
    __syncthreads();
    if (threadIdx.x == 0) ring_drain(rx, full, PS::kStages, consumed, p.wait_cycles, p.status);
}

}  // namespace

// Number of SMs of the current device (cached per device).
static int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Opt in to the ring's shared memory and read how many CTAs of the kernel an
// SM of this device holds (cached per device).
template <typename TS, int L>
static cudaError_t resident_ctas(int *ctas) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        using PS = PackedPipe<TS, L>;
        e = cudaFuncSetAttribute(ssu_packed_kernel<TS, L>, cudaFuncAttributeMaxDynamicSharedMemorySize, PS::kBytes);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ssu_packed_kernel<TS, L>, PS::kThreads, PS::kBytes);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorInvalidConfiguration;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    *ctas = n;
    return cudaSuccess;
}

template <typename TS, int L>
static cudaError_t launch_t(const KParams &p, cudaStream_t stream) {
    using PS = PackedPipe<TS, L>;
    int per_sm = 0;
    cudaError_t e = resident_ctas<TS, L>(&per_sm);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t units = p.nseq * p.H * p.ptiles;
    const int64_t slots_on_gpu = static_cast<int64_t>(sms) * per_sm;
    const int64_t grid = units < slots_on_gpu ? units : slots_on_gpu;
    ssu_packed_kernel<TS, L><<<static_cast<unsigned>(grid), PS::kThreads, PS::kBytes, stream>>>(p);
    return cudaGetLastError();
}

template <typename TS>
static cudaError_t launch_lanes(int lanes, const KParams &p, cudaStream_t stream) {
    switch (lanes) {
    case 1: return launch_t<TS, 1>(p, stream);
    case 2: return launch_t<TS, 2>(p, stream);
    case 4: return launch_t<TS, 4>(p, stream);
    case 8: return launch_t<TS, 8>(p, stream);
    case 16: return launch_t<TS, 16>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_packed(int state_dtype, int lanes, const KParams &p, cudaStream_t stream) {
    if (p.rows >= kLongRowsPerSeq * p.nseq) return launch_packed_long(state_dtype, lanes, p, stream);
    switch (state_dtype) {
    case kF32: return launch_lanes<float>(lanes, p, stream);
    case kF16: return launch_lanes<__half>(lanes, p, stream);
    case kBF16: return launch_lanes<__nv_bfloat16>(lanes, p, stream);
    }
    return cudaErrorInvalidValue;
}

template <typename TS, int L>
static cudaError_t attrs_t() {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, ssu_packed_kernel<TS, L>);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if (sm_count() <= 0) return cudaErrorInvalidDevice;
    return resident_ctas<TS, L>(&per_sm);
}

template <typename TS>
static cudaError_t attrs_lanes(int lanes) {
    switch (lanes) {
    case 1: return attrs_t<TS, 1>();
    case 2: return attrs_t<TS, 2>();
    case 4: return attrs_t<TS, 4>();
    case 8: return attrs_t<TS, 8>();
    case 16: return attrs_t<TS, 16>();
    }
    return cudaErrorInvalidValue;
}

cudaError_t prewarm_packed(int state_dtype, int lanes) {
    const cudaError_t e = prewarm_packed_long(state_dtype, lanes);
    if (e != cudaSuccess) return e;
    switch (state_dtype) {
    case kF32: return attrs_lanes<float>(lanes);
    case kF16: return attrs_lanes<__half>(lanes);
    case kBF16: return attrs_lanes<__nv_bfloat16>(lanes);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ssu
