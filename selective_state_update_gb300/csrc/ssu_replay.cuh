// ssu_replay.cuh -- decode on the checkpoint + buffer form of the state.
//
// Article "ReplaySSM: Cache SSM Inputs, Not State", section 核心做法: the
// state of a slot is a checkpoint plus the inputs (v, dt', k) = (x, dt', B) of
// the steps since the last fold.  Unrolled, the state after the current step
// c is
//     S_c = gamma_{0:c} S_ckpt + sum_{j<=c} gamma_{j+1:c} dt'_j x_j B_j^T,
//     gamma_{i:c} = prod_{m=i..c} exp(A dt'_m),
// so y = S_c . C can be read out without forming S_c:
//     y = gamma_{0:c} (S_ckpt . C) + sum_j gamma_{j+1:c} dt'_j x_j (B_j . C).
// A step that does not fill the buffer does exactly that and appends its
// inputs; the checkpoint is read but not written.  The step that fills it
// folds the entries into the checkpoint in order (the plain update, carried in
// fp32, with the plain kernels' decays bit for bit), reads y out of the result
// and writes the checkpoint back once.  Section 数据与边界: the checkpoint is
// read every step and written once every L steps, so the state traffic per
// step drops from a read and a write to about a read.
//
// Work unit: (sequence b, head h, tile of kTileRows dim rows), numbered as in
// the one-token kernel.  The kernel is persistent and warp-specialised, with a
// ring of shared-memory stages per CTA:
//   producer warps  one unit each in turn, operands loaded a unit ahead:
//                   resolve the slot and the buffered count c, write the
//                   count for the next step, compute the current token's row
//                   scalars {dA, dt' x, x, gate} into the stage, append its
//                   entry (x, dt', and B once per group) when the buffer does
//                   not fill, stage B and C, and request the checkpoint tile
//                   and the c buffered entries of the tile (x rows, dt' rows,
//                   B of the group) as bulk asynchronous copies (TMA engine)
//                   completing on the stage's "full" mbarrier;
//   consumer warps  either the readout -- S_ckpt . C per row beside the B_j . C
//                   dots (one warp per dot), then the walk over the entries,
//                   split in contiguous parts over the lanes of a row and
//                   combined by shuffles, and y -- or the fold -- each entry's
//                   decay and input term per row, the entries in order, then
//                   the current token; y; the tile back into the stage, from
//                   where one thread stores it to the checkpoint with a bulk
//                   copy.  A stage is released on its "empty"
//                   mbarrier once read, or once its store has read it out.
// The kernel is compiled per dtype of the 16/32-bit operands (IO), which
// keeps the consumer's code small and free of dtype branches.
#pragma once

#include <atomic>

#include "ssu_device.cuh"

namespace ssu {

// Most stages of a ring.
constexpr int kReplayMaxStages = 6;
static_assert(kReplayMaxStages <= kMaxRingStages, "ring exit record too small");
// Size of the pieces the checkpoint tile is requested in (lanes in turn).
constexpr uint32_t kReplayTileChunk = 32768;

template <typename TS, int L, int SH = kShadowNone>
struct ReplayPipe {
    // State rows per consumer thread: four, as in the plain kernels, or two
    // when the consumers decode an NVFP4 copy, so that its decode and the
    // unit's short dependent phases run on twice the warps (measured: NVFP4
    // 0.358 ms against 0.416 ms with four; fp32 0.331 against 0.294, where the
    // 96-register budget of two costs more than the warps gain).  Four at
    // dstate 256 in any case.
    static constexpr int kRows = SH == kShadowNVFP4 && L < 16 ? 2 : 4;
    static constexpr int kSlots = kTileRows / kRows;
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kTileBytes = kTileRows * kN * static_cast<int>(sizeof(TS));
    static constexpr int kConsumerWarps = (kSlots * L + 31) / 32;
    static constexpr int kConsumers = 32 * kConsumerWarps;
    // Producer warps take units in turn; a producer waits for its stage by
    // the parity of the "empty" phase, which is unambiguous only with no more
    // producers than stages, so a one-stage ring runs one producer.
    static constexpr int kProducerWarps = 2;
    static constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
    // Where the E4M3 row scales of a read copy sit in a stage: after the
    // largest copy tile (one byte per element), inside the checkpoint tile.
    static constexpr int kShadowScaleOffset = kTileRows * kN;
    static_assert(kShadowScaleOffset + kTileRows * 4 <= kTileBytes, "read-copy scales do not fit the tile");
    // Where the NVFP4 scale records sit: after the largest tile of code pairs.
    static constexpr int kNvfp4RecOffset = kTileRows * kN / 2;
    static_assert(kNvfp4RecOffset + kTileRows * nvfp4_scale_words(kN) * 4 <= kTileBytes,
                  "NVFP4 scale records do not fit the tile");
    // Register budget: two CTAs per SM where a tile and a few KB of entries
    // fit twice in half of an SM's shared memory (228 KB on this part, less a
    // margin) and two CTAs still leave 128 registers a thread.  The ring
    // itself is sized at launch from the device's shared memory per SM.
    static constexpr int kMinCtas =
        (222 * 1024 / 2 - 1024) / (kTileBytes + 4096) >= 2 && 65536 / (2 * kThreads) >= 96 ? 2 : 1;
};

// Per-stage header written by the producer.
struct ReplayHeader {
    int64_t slot;
    int32_t flags;  // kR* bits
    int32_t c;      // buffered entries of the slot (0 for a pad slot)
    float Dh, Ah;
    int32_t reserved[2];
};
enum : int32_t { kRValid = 1, kRSeeded = 2, kRFold = 4 };

// Stage strides (elements) between the buffered entries' x rows and dt'
// rows: a tile's rows plus 16 bytes, so that the lanes of a row, which read
// neighbouring entries of the same row at once, fall in different banks.
template <int IO>
__host__ __device__ constexpr int x_stride() { return kTileRows + (IO == kF32 ? 4 : 8); }
constexpr int kDtStride = kTileRows + 4;

// Shared-memory layout, fixed per launch by the buffer length and the size of
// the 16/32-bit operands.  A stage holds the checkpoint tile, up to len - 1
// buffered entries as stored (x rows and dt' rows of the tile, B of the
// group), the current token's B and C as fp32, the row scalars and the
// header.  After the ring: the CTA's scratch for the unit being computed (B .
// C dots; per-entry decays and input terms of a fold) and the mbarriers.
struct ReplayLayout {
    int xe, de, be, bc, cs, rowq, hd, stage;
    int stages, producers, dots, rowa, rowb, bars, exit, bytes, ctas;

    __host__ __device__ static int up(int v) { return (v + 127) / 128 * 128; }

    __host__ __device__ void place(int tile_bytes, int n, int len, int io) {
        const int ent = len - 1;
        const int xs = kTileRows + 16 / io;
        xe = up(tile_bytes);                 // io  [ent][xs]
        de = up(xe + ent * xs * io);         // f32 [ent][kDtStride]
        be = up(de + ent * kDtStride * 4);   // io  [ent][n]
        bc = up(be + ent * n * io);          // f32 [n]
        cs = bc + n * 4;                     // f32 [n]
        rowq = up(cs + n * 4);               // f32x4 [kTileRows]
        hd = rowq + kTileRows * 16;          // ReplayHeader
        stage = up(hd + static_cast<int>(sizeof(ReplayHeader)));
    }
    // Ring of `stages` stages followed by the scratch and the barriers.
    __host__ __device__ void finish(int len) {
        dots = stages * stage;                                 // f32 [len]
        rowa = up(dots + len * 4);                             // f32 [len - 1][kTileRows]
        rowb = up(rowa + (len - 1) * kTileRows * 4);           // f32 [len - 1][kTileRows]
        bars = up(rowb + (len - 1) * kTileRows * 4);           // u64 full[stages], empty[stages]
        exit = bars + 2 * 8 * stages;                          // RingExit
        bytes = exit + static_cast<int>(sizeof(RingExit));
    }
    static int scratch(int len) {
        return up(len * 4) + 2 * up((len - 1) * kTileRows * 4) + 2 * 8 * kReplayMaxStages +
               static_cast<int>(sizeof(RingExit));
    }
    // Two CTAs per SM when registers allow two (max_ctas) and each still gets
    // a ring of two stages, else one CTA with as many stages as fit (at most
    // kReplayMaxStages; a single stage -- fp32 checkpoints of dstate 256 with
    // long fp32 buffers -- runs without overlap).  `smem_per_sm` is what the
    // CTAs of an SM may take in all.  Returns false when not even one stage
    // fits.
    bool choose(int tile_bytes, int n, int len, int io, int smem_per_sm, int max_ctas, int max_producers) {
        place(tile_bytes, n, len, io);
        const int sc = scratch(len);
        auto fit = [&](int k) { return (smem_per_sm / k - 1024 - sc) / stage; };
        ctas = max_ctas >= 2 && fit(2) >= 2 ? 2 : 1;
        stages = fit(ctas);
        if (stages > kReplayMaxStages) stages = kReplayMaxStages;
        if (stages < 1) return false;
        producers = stages < max_producers ? stages : max_producers;
        finish(len);
        return true;
    }
};

// Element i of a buffer stored in the io dtype IO, as fp32.
template <int IO>
__device__ __forceinline__ float io_at(const unsigned char *base, int i) {
    if constexpr (IO == kF32)
        return reinterpret_cast<const float *>(base)[i];
    else
        return bits_to_float(reinterpret_cast<const unsigned short *>(base)[i], IO);
}

// This thread's 16 values of one buffered B entry (stored in the io dtype),
// as fp32, in the element layout of Tile::gather: vector loads of each
// thread's contiguous chunks.
template <typename TS, int L, int IO>
__device__ __forceinline__ void gather_entry(const unsigned char *row, int lane, float *v) {
    using T = Tile<TS, L>;
    constexpr int V = T::kVec;
#pragma unroll
    for (int k = 0; k < T::kChunks; ++k) {
        const int off = (lane + L * k) * V;
        if constexpr (IO == kF32) {
#pragma unroll
            for (int q = 0; q < V / 4; ++q) {
                const float4 f = reinterpret_cast<const float4 *>(row)[off / 4 + q];
                v[k * V + 4 * q + 0] = f.x;
                v[k * V + 4 * q + 1] = f.y;
                v[k * V + 4 * q + 2] = f.z;
                v[k * V + 4 * q + 3] = f.w;
            }
        } else {
            uint32_t w[V / 2];
            if constexpr (V == 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(row + off * 2);
                w[0] = u.x;
                w[1] = u.y;
                w[2] = u.z;
                w[3] = u.w;
            } else {
                const uint2 u = *reinterpret_cast<const uint2 *>(row + off * 2);
                w[0] = u.x;
                w[1] = u.y;
            }
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                v[k * V + 2 * i] = bits_to_float(w[i] & 0xffffu, IO);
                v[k * V + 2 * i + 1] = bits_to_float(w[i] >> 16, IO);
            }
        }
    }
}

// V consecutive elements of a buffer stored in the io dtype IO, as fp32, with
// one vector load (V * sizeof <= 16 bytes, aligned).
template <int IO, int V>
__device__ __forceinline__ void io_vec(const unsigned char *base, int i, float *v) {
    if constexpr (IO == kF32) {
        static_assert(V == 2 || V == 4, "fp32 vectors of 2 or 4");
        if constexpr (V == 4) {
            const float4 f = reinterpret_cast<const float4 *>(base)[i / 4];
            v[0] = f.x, v[1] = f.y, v[2] = f.z, v[3] = f.w;
        } else {
            const float2 f = reinterpret_cast<const float2 *>(base)[i / 2];
            v[0] = f.x, v[1] = f.y;
        }
    } else {
        static_assert(V == 2 || V == 4 || V == 8, "16-bit vectors of 2, 4 or 8");
        uint32_t w[V / 2];
        if constexpr (V == 8) {
            const uint4 u = reinterpret_cast<const uint4 *>(base)[i / 8];
            w[0] = u.x, w[1] = u.y, w[2] = u.z, w[3] = u.w;
        } else if constexpr (V == 4) {
            const uint2 u = reinterpret_cast<const uint2 *>(base)[i / 4];
            w[0] = u.x, w[1] = u.y;
        } else {
            w[0] = reinterpret_cast<const uint32_t *>(base)[i / 2];
        }
#pragma unroll
        for (int k = 0; k < V / 2; ++k) {
            v[2 * k] = bits_to_float(w[k] & 0xffffu, IO);
            v[2 * k + 1] = bits_to_float(w[k] >> 16, IO);
        }
    }
}

// B_j . C for the c buffered entries (j < c) and the current token (j = c):
// eight lanes per dot, kConsumers / 8 dots at a time.  Lane s of a dot takes
// the chunks s, s + 8, ... of V elements (V * sizeof(io) <= 16 bytes), so a
// warp's loads of one chunk index cover whole 128-byte lines per dot.
template <int N, int kConsumers, int IO>
__device__ __forceinline__ void entry_dots(int c, const unsigned char *be, const float *sB, const float *sC,
                                           float *dots, int tid) {
    constexpr int kIo = IO == kF32 ? 4 : 2;
    constexpr int kPer = N / 8;                                   // elements per lane
    constexpr int V = kPer < 16 / kIo ? kPer : 16 / kIo;          // elements per chunk
    constexpr int kChunks = kPer / V;
    constexpr int kDots = kConsumers / 8;
    static_assert(kPer % V == 0 && V >= 2, "dstate must be a multiple of 16");
    const int grp = tid / 8, seg = tid % 8;
    float cv[kPer];
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
        const int n = (seg + 8 * k) * V;
#pragma unroll
        for (int v = 0; v < V; ++v) cv[k * V + v] = sC[n + v];
    }
    for (int base = 0; base <= c; base += kDots) {  // same trip count for every thread
        const int j = base + grp;
        float acc[2] = {0.f, 0.f};
        if (j < c) {
#pragma unroll
            for (int k = 0; k < kChunks; ++k) {
                float bv[V];
                io_vec<IO, V>(be, j * N + (seg + 8 * k) * V, bv);
#pragma unroll
                for (int v = 0; v < V; ++v) acc[v & 1] = fmaf(bv[v], cv[k * V + v], acc[v & 1]);
            }
        } else if (j == c) {
#pragma unroll
            for (int k = 0; k < kChunks; ++k) {
                const int n = (seg + 8 * k) * V;
#pragma unroll
                for (int v = 0; v < V; ++v) acc[v & 1] = fmaf(sB[n + v], cv[k * V + v], acc[v & 1]);
            }
        }
        float d = acc[0] + acc[1];
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        if (seg == 0 && j <= c) dots[j] = d;
    }
}

// Each buffered entry's decay exp(A dt'_j) and input term dt'_j x_j for every
// row of the tile, into rowa / rowb ([entry][kTileRows]), for a fold; loads
// of a batch issued before its arithmetic.  The decays come from the plain
// kernels' function, so that the folded state is theirs bit for bit.
template <int kThreads, int IO>
__device__ __forceinline__ void entry_terms(int c, int rows, float Ah, const float *de, const unsigned char *xe,
                                            float *rowa, float *rowb, int tid) {
    constexpr int kB = 4;
    const int total = c * kTileRows;
    for (int i0 = tid; i0 < total; i0 += kB * kThreads) {
        float d[kB], x[kB];
#pragma unroll
        for (int q = 0; q < kB; ++q) {
            const int i = i0 + q * kThreads;
            const int j = i / kTileRows, r = i % kTileRows;
            const bool ok = i < total && r < rows;
            d[q] = ok ? de[j * kDtStride + r] : 0.f;
            x[q] = ok ? io_at<IO>(xe, j * x_stride<IO>() + r) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kB; ++q) {
            const int i = i0 + q * kThreads;
            if (i < total && i % kTileRows < rows) {
                rowa[i] = decay(Ah, d[q]);
                rowb[i] = d[q] * x[q];
            }
        }
    }
}

// This thread's 16 values of row rr of a read copy staged in shared memory
// (E4M3 codes times nothing, or E2M1 codes times their block scale -- the
// caller applies the row scale -- or fp16), in the element layout of
// Tile::gather.
template <typename TS, int L>
__device__ __forceinline__ void load_copy_row(const unsigned char *tile, int rr, int lane, int fmt, float *v) {
    using T = Tile<TS, L>;
    constexpr int V = T::kVec;
    constexpr int N = T::kN;
#pragma unroll
    for (int k = 0; k < T::kChunks; ++k) {
        const int e0 = (lane + L * k) * V;
        if (fmt == kShadowNVFP4) {
            const unsigned char *rec = tile + kTileRows * N / 2 + rr * nvfp4_scale_words(N) * 4;
            const float bs = e4m3_value(rec[4 + e0 / 16]);
            uint32_t w;
            if constexpr (V == 8)
                w = *reinterpret_cast<const uint32_t *>(tile + rr * (N / 2) + e0 / 2);
            else
                w = *reinterpret_cast<const unsigned short *>(tile + rr * (N / 2) + e0 / 2);
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                const float2 f = e2m1x2_values(w >> (8 * i));
                v[k * V + 2 * i] = f.x * bs;
                v[k * V + 2 * i + 1] = f.y * bs;
            }
        } else if (fmt == kShadowE4M3) {
            uint32_t w[V / 4];
            if constexpr (V == 8) {
                const uint2 u = *reinterpret_cast<const uint2 *>(tile + rr * N + e0);
                w[0] = u.x, w[1] = u.y;
            } else {
                w[0] = *reinterpret_cast<const uint32_t *>(tile + rr * N + e0);
            }
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                const float2 f = e4m3x2_values(w[i / 2] >> (16 * (i % 2)));
                v[k * V + 2 * i] = f.x;
                v[k * V + 2 * i + 1] = f.y;
            }
        } else {
            uint32_t w[V / 2];
            const unsigned char *src = tile + (rr * N + e0) * 2;
            if constexpr (V == 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(src);
                w[0] = u.x, w[1] = u.y, w[2] = u.z, w[3] = u.w;
            } else {
                const uint2 u = *reinterpret_cast<const uint2 *>(src);
                w[0] = u.x, w[1] = u.y;
            }
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                v[k * V + 2 * i] = bits_to_float(w[i] & 0xffffu, kF16);
                v[k * V + 2 * i + 1] = bits_to_float(w[i] >> 16, kF16);
            }
        }
    }
}

// Writes the read copy of one folded state row (this thread's 16 values `sv`
// as the pool stores them) to global memory: E4M3 codes and the row scale,
// NVFP4 codes and the row's scale record, or fp16.  Every lane of the row
// takes part (the row and block maxima are shuffles); only `live` rows are
// written.
template <typename TS, int L, int SH>
__device__ __forceinline__ void write_copy_row(const KParams &p, int64_t row, int lane, bool live, const float *sv) {
    using T = Tile<TS, L>;
    constexpr int V = T::kVec;
    constexpr int N = T::kN;
    float st[kElemsPerThread];
    if constexpr (sizeof(TS) == 4) {
#pragma unroll
        for (int i = 0; i < kElemsPerThread; ++i) st[i] = sv[i];
    } else {
#pragma unroll
        for (int k = 0; k < T::kChunks; ++k) StateChunk<TS>::unpack(StateChunk<TS>::pack(sv + k * V), st + k * V);
    }
    if constexpr (SH == kShadowE4M3) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < kElemsPerThread; ++i) amax = fmaxf(amax, fabsf(st[i]));
#pragma unroll
        for (int off = L / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float sc = shadow_scale_of(amax), f = shadow_factor_of(amax);
        if (!live) return;
        unsigned char *out = static_cast<unsigned char *>(p.shadow) + row * N;
#pragma unroll
        for (int k = 0; k < T::kChunks; ++k) {
            uint32_t w[V / 4] = {};
#pragma unroll
            for (int i = 0; i < V / 2; ++i)
                w[i / 2] |= e4m3x2_codes(__fmul_rn(st[k * V + 2 * i], f), __fmul_rn(st[k * V + 2 * i + 1], f))
                            << (16 * (i % 2));
            unsigned char *dst = out + (lane + L * k) * V;
            if constexpr (V == 8)
                *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
            else
                *reinterpret_cast<uint32_t *>(dst) = w[0];
        }
        if (lane == 0) p.shadow_scale[row] = sc;
    } else if constexpr (SH == kShadowNVFP4) {
        // a block of 16 elements is G neighbouring lanes' chunks (same k)
        constexpr int G = 16 / V;
        static_assert(L % G == 0, "an NVFP4 block must lie within one row's lanes");
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < kElemsPerThread; ++i) amax = fmaxf(amax, fabsf(st[i]));
#pragma unroll
        for (int off = L / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float sr = nvfp4_row_scale(amax);
        uint32_t w[T::kChunks], bc[T::kChunks];
#pragma unroll
        for (int k = 0; k < T::kChunks; ++k) {
            float bmax = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) bmax = fmaxf(bmax, fabsf(st[k * V + i]));
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
            bc[k] = nvfp4_block_code(bmax, sr);
            const float den = __fmul_rn(e4m3_value(bc[k]), sr);
            w[k] = 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                const float q0 = den > 0.f ? __fdiv_rn(st[k * V + 2 * i], den) : 0.f;
                const float q1 = den > 0.f ? __fdiv_rn(st[k * V + 2 * i + 1], den) : 0.f;
                w[k] |= e2m1x2_code(q0, q1) << (8 * i);
            }
        }
        if (!live) return;
        unsigned char *out = static_cast<unsigned char *>(p.shadow) + row * (N / 2);
        unsigned char *rec = reinterpret_cast<unsigned char *>(p.shadow_scale + row * nvfp4_scale_words(N));
#pragma unroll
        for (int k = 0; k < T::kChunks; ++k) {
            const int e0 = (lane + L * k) * V;
            if constexpr (V == 8)
                *reinterpret_cast<uint32_t *>(out + e0 / 2) = w[k];
            else
                *reinterpret_cast<unsigned short *>(out + e0 / 2) = static_cast<unsigned short>(w[k]);
            if (lane % G == 0) rec[4 + e0 / 16] = static_cast<unsigned char>(bc[k]);
        }
        if (lane == 0) *reinterpret_cast<float *>(rec) = sr;
    } else if (SH == kShadowF16 && live) {
        unsigned char *out = static_cast<unsigned char *>(p.shadow) + row * N * 2;
#pragma unroll
        for (int k = 0; k < T::kChunks; ++k) {
            uint32_t w[V / 2];
#pragma unroll
            for (int i = 0; i < V / 2; ++i)
                w[i] = uint32_t(__half_as_ushort(__float2half_rn(st[k * V + 2 * i]))) |
                       (uint32_t(__half_as_ushort(__float2half_rn(st[k * V + 2 * i + 1]))) << 16);
            unsigned char *dst = out + (lane + L * k) * V * 2;
            if constexpr (V == 8)
                *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            else
                *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
        }
    }
}

// The operands of one unit plus its slot's buffered count (lane 0).
template <typename TS, int L>
struct ReplayOperands : UnitOperands<TS, L> {
    int cnt;
    __device__ __forceinline__ void load(const KParams &p, const UnitCoords &cu, int lane) {
        UnitOperands<TS, L>::load(p, cu, lane);
        cnt = lane == 0 ? __ldg(p.cnt_in + cu.b) : 0;
    }
};

// Stage one unit (see the file comment).  Returns false on a timed-out wait.
template <typename TS, int L, int IO, int SH>
__device__ __forceinline__ bool produce_replay(const KParams &p, const ReplayLayout &lay,
                                               const ReplayOperands<TS, L> &op, int k, unsigned char *smem,
                                               uint64_t *full, uint64_t *empty, RingExit *rx, int lane) {
    constexpr int N = ReplayPipe<TS, L>::kN;
    constexpr int io = IO == kF32 ? 4 : 2;
    constexpr int kPerB = UnitOperands<TS, L>::kPerB;
    constexpr int kPerRow = UnitOperands<TS, L>::kPerRow;
    const int S = lay.stages;
    const int s = k % S;
    const int round = k / S;
    const int len = p.rlen;
    const UnitCoords &cu = op.c;

    // First everything that does not touch the stage, while the consumers
    // may still hold it: the unit's flags and count, the current token's row
    // scalars (the same calls the plain kernels make: bit-identical), and its
    // appended entry.
    int32_t flags = 0, c = 0;
    if (lane == 0) {
        if (op.entries_ok && slot_ok(p, op.rs)) {
            if (op.rs == p.pad) {
                flags = kRValid | kRFold;  // zero state, nothing buffered, nothing written
            } else if (op.cnt < 0 || op.cnt >= len) {
                flag(p.status, kDevBadCount);
            } else {
                c = op.cnt;
                flags = kRValid | kRSeeded | (c + 1 == len ? kRFold : 0);
            }
        }
        if ((flags & kRValid) && cu.h == 0 && cu.row0 == 0) p.cnt_out[cu.b] = (flags & kRFold) ? 0 : c + 1;
    }
    flags = __shfl_sync(0xffffffffu, flags, 0);
    c = __shfl_sync(0xffffffffu, c, 0);
    const int64_t rs = __shfl_sync(0xffffffffu, op.rs, 0);
    const bool append = (flags & kRValid) && !(flags & kRFold);
    if (append && cu.h % p.heads_per_group == 0 && cu.row0 == 0) {
#pragma unroll
        for (int i = 0; i < kPerB; ++i) {
            const int n = lane + 32 * i;
            if (n < N) {
                const int64_t e = ((rs * len + c) * p.G + cu.g) * static_cast<int64_t>(N) + n;
                if constexpr (io == 4)
                    static_cast<unsigned int *>(p.Bbuf)[e] = op.b[i];
                else
                    static_cast<unsigned short *>(p.Bbuf)[e] = static_cast<unsigned short>(op.b[i]);
            }
        }
    }
    float4 rq[kPerRow];
#pragma unroll
    for (int i = 0; i < kPerRow; ++i) {
        const int r = lane + 32 * i;
        rq[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < cu.rows_here && (flags & kRValid)) {
            const float xv = bits_to_float(op.x[i], IO);
            const float d = processed_step(bits_to_float(op.dt[i], p.dt_dtype), op.bias, p.softplus);
            rq[i] = make_float4(decay(op.Ah, d), d * xv, xv, silu_gate(bits_to_float(op.z[i], IO), p.z != nullptr));
            if (append) {
                const int64_t e = ((rs * len + c) * p.H + cu.h) * static_cast<int64_t>(p.P) + cu.row0 + r;
                p.dtbuf[e] = d;
                if constexpr (io == 4)
                    static_cast<unsigned int *>(p.xbuf)[e] = op.x[i];
                else
                    static_cast<unsigned short *>(p.xbuf)[e] = static_cast<unsigned short>(op.x[i]);
            }
        }
    }

    // Then the stage: header, B, C, row scalars, the copies.
    if (ring_aborted(rx)) return false;
    if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1, p.wait_cycles)) {
        if (lane == 0) {
            flag(p.status, kDevTimeout);
            ring_abort(rx);
        }
        return false;
    }
    unsigned char *base = smem + s * lay.stage;
    ReplayHeader *hd = reinterpret_cast<ReplayHeader *>(base + lay.hd);
    float *sB = reinterpret_cast<float *>(base + lay.bc);
    float *sC = reinterpret_cast<float *>(base + lay.cs);
    float4 *rowq = reinterpret_cast<float4 *>(base + lay.rowq);
    if (lane == 0) {
        hd->slot = op.rs;
        hd->flags = flags;
        hd->c = c;
        hd->Dh = op.Dh;
        hd->Ah = op.Ah;
    }
#pragma unroll
    for (int i = 0; i < kPerB; ++i) {
        const int n = lane + 32 * i;
        if (n < N) {
            sB[n] = bits_to_float(op.b[i], IO);
            sC[n] = bits_to_float(op.cc[i], IO);
        }
    }
#pragma unroll
    for (int i = 0; i < kPerRow; ++i) {
        const int r = lane + 32 * i;
        if (r < cu.rows_here) rowq[r] = rq[i];
    }

    if (!(flags & kRSeeded)) {
        mbar_arrive(&full[s]);
        return true;
    }
    unsigned char *xe = base + lay.xe;
    float *de = reinterpret_cast<float *>(base + lay.de);
    unsigned char *be = base + lay.be;
    const int rows = cu.rows_here;
    const bool bulk_entries = p.rbulk != 0;
    if (!bulk_entries) {
        // Buffers not 16-byte aligned: plain loads of the same entries.
        for (int i = lane; i < c * rows; i += 32) {
            const int j = i / rows, r = i % rows;
            const int64_t e = ((rs * len + j) * p.H + cu.h) * static_cast<int64_t>(p.P) + cu.row0 + r;
            de[j * kDtStride + r] = __ldg(p.dtbuf + e);
            if constexpr (io == 4)
                reinterpret_cast<unsigned int *>(xe)[j * x_stride<IO>() + r] = load_bits<true>(p.xbuf, e);
            else
                reinterpret_cast<unsigned short *>(xe)[j * x_stride<IO>() + r] =
                    static_cast<unsigned short>(load_bits<false>(p.xbuf, e));
        }
        for (int i = lane; i < c * N; i += 32) {
            const int j = i / N, n = i % N;
            const int64_t e = ((rs * len + j) * p.G + cu.g) * static_cast<int64_t>(N) + n;
            if constexpr (io == 4)
                reinterpret_cast<unsigned int *>(be)[j * N + n] = load_bits<true>(p.Bbuf, e);
            else
                reinterpret_cast<unsigned short *>(be)[j * N + n] = static_cast<unsigned short>(load_bits<false>(p.Bbuf, e));
        }
    }
    // The checkpoint tile and (aligned buffers) every buffered entry, as bulk
    // copies; lane 0 registers the total before any copy can complete.  (One
    // copy per entry and buffer measured faster than one run per buffer of a
    // head-major buffer layout.)
    // A step that does not fold reads the read copy when there is one
    // (codes, then E4M3 row scales at kShadowScaleOffset), else the tile.
    const bool read_copy = SH != kShadowNone && !(flags & kRFold);
    const int64_t row_first = (rs * p.H + cu.h) * static_cast<int64_t>(p.P) + cu.row0;
    // bytes of one row of the tile as requested: the read copy's codes or the checkpoint
    const uint32_t row_bytes = !read_copy ? N * sizeof(TS)
                               : SH == kShadowF16 ? N * 2 : SH == kShadowNVFP4 ? N / 2 : N;
    const uint32_t tile_bytes = static_cast<uint32_t>(rows) * row_bytes;
    const uint32_t scale_bytes = !read_copy ? 0
                                 : SH == kShadowE4M3 ? static_cast<uint32_t>(rows) * 4
                                 : SH == kShadowNVFP4 ? static_cast<uint32_t>(rows) * nvfp4_scale_words(N) * 4 : 0;
    uint32_t bytes = tile_bytes + scale_bytes;
    if (bulk_entries) bytes += static_cast<uint32_t>(c) * (rows * (io + 4) + N * io);
    if (lane == 0) mbar_arrive_expect(&full[s], bytes);
    __syncwarp();
    if (scale_bytes != 0 && lane == 31) {
        if constexpr (SH == kShadowNVFP4)
            bulk_load(base + ReplayPipe<TS, L>::kNvfp4RecOffset, p.shadow_scale + row_first * nvfp4_scale_words(N),
                      scale_bytes, &full[s]);
        else
            bulk_load(base + ReplayPipe<TS, L>::kShadowScaleOffset, p.shadow_scale + row_first, scale_bytes, &full[s]);
    }
    {
        const unsigned char *src =
            read_copy ? static_cast<const unsigned char *>(p.shadow) + row_first * row_bytes
                      : reinterpret_cast<const unsigned char *>(static_cast<const TS *>(p.state) + row_first * N);
        for (uint32_t off = static_cast<uint32_t>(lane) * kReplayTileChunk; off < tile_bytes;
             off += 32u * kReplayTileChunk)
            bulk_load(base + off, src + off, tile_bytes - off < kReplayTileChunk ? tile_bytes - off : kReplayTileChunk,
                      &full[s]);
    }
    if (bulk_entries) {
        for (int j = lane; j < c; j += 32) {
            const int64_t e = ((rs * len + j) * p.H + cu.h) * static_cast<int64_t>(p.P) + cu.row0;
            bulk_load(xe + j * x_stride<IO>() * io, static_cast<const unsigned char *>(p.xbuf) + e * io,
                      static_cast<uint32_t>(rows) * io, &full[s]);
            bulk_load(de + j * kDtStride, p.dtbuf + e, static_cast<uint32_t>(rows) * 4, &full[s]);
            const int64_t eb = ((rs * len + j) * p.G + cu.g) * static_cast<int64_t>(N);
            bulk_load(be + j * N * io, static_cast<const unsigned char *>(p.Bbuf) + eb * io,
                      static_cast<uint32_t>(N) * io, &full[s]);
        }
    }
    if (lane == 0) ring_note_fill(rx, s, round);
    if (lane != 0) mbar_arrive(&full[s]);
    return true;
}

// Producer warp `w` stages the CTA's units k = w, w + P, w + 2P, ...
// (P = lay.producers), i.e. global units blockIdx.x + k * gridDim.x.
template <typename TS, int L, int IO, int SH>
__device__ __forceinline__ void replay_producer(const KParams &p, const ReplayLayout &lay, int64_t units,
                                                unsigned char *smem, uint64_t *full, uint64_t *empty, RingExit *rx,
                                                int w) {
    const int P = lay.producers;
    if (w >= P) return;
    const int lane = threadIdx.x & 31;
    const int64_t step = static_cast<int64_t>(P) * gridDim.x;
    ReplayOperands<TS, L> a, b;
    int64_t u = blockIdx.x + static_cast<int64_t>(w) * gridDim.x;
    UnitWalker walk(p, u, step);
    if (u < units) a.load(p, walk.coords(p), lane);
    for (int k = w; u < units; k += 2 * P, u += 2 * step) {
        walk.advance(p);
        if (u + step < units) b.load(p, walk.coords(p), lane);
        if (!produce_replay<TS, L, IO, SH>(p, lay, a, k, smem, full, empty, rx, lane)) return;
        if (u + step >= units) break;
        walk.advance(p);
        if (u + 2 * step < units) a.load(p, walk.coords(p), lane);
        if (!produce_replay<TS, L, IO, SH>(p, lay, b, k + P, smem, full, empty, rx, lane)) return;
    }
}

// Returns the ring index of the first unit not consumed.
template <typename TS, int L, int IO, int SH>
__device__ __forceinline__ int replay_consumer(const KParams &p, const ReplayLayout &lay, int64_t units,
                                               unsigned char *smem, uint64_t *full, uint64_t *empty, RingExit *rx) {
    using T = Tile<TS, L>;
    using PS = ReplayPipe<TS, L, SH>;
    constexpr int N = PS::kN;
    constexpr int kConsumers = PS::kConsumers;
    constexpr int io = IO == kF32 ? 4 : 2;
    const int S = lay.stages;
    const int tid = threadIdx.x;
    constexpr int kReplayRows = PS::kRows, kReplaySlots = PS::kSlots;
    const bool active = tid < kReplaySlots * L;
    const int lane = tid % L;
    const int slot_row = tid / L;
    float *dots = reinterpret_cast<float *>(smem + lay.dots);
    float *rowa = reinterpret_cast<float *>(smem + lay.rowa);
    float *rowb = reinterpret_cast<float *>(smem + lay.rowb);
    int pending = -1;  // stage whose checkpoint store may still be reading it (thread 0)
    int k = 0;
    UnitWalker walk(p, blockIdx.x, gridDim.x);
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++k, walk.advance(p)) {
        const int s = k % S;
        const bool ok = mbar_wait_bounded(&full[s], (k / S) & 1, p.wait_cycles);
        if (barrier_or(1, kConsumers, !ok)) {  // a wait gave up: every consumer stops here
            if (tid == 0) {
                flag(p.status, kDevTimeout);
                ring_abort(rx);
                bulk_wait_all();
            }
            return k;
        }
        unsigned char *base = smem + s * lay.stage;
        const ReplayHeader *hd = reinterpret_cast<const ReplayHeader *>(base + lay.hd);
        const int32_t flags = hd->flags;
        const bool fold = (flags & kRFold) != 0;
        const bool seeded = (flags & kRSeeded) != 0;
        const bool stores = (flags & kRValid) && fold && seeded;
        const UnitCoords cu = walk.coords(p);
        if (flags & kRValid) {
            const int c = hd->c;
            const int rows = cu.rows_here;
            const float Ah = hd->Ah, Dh = hd->Dh;
            TS *tile = reinterpret_cast<TS *>(base);
            const unsigned char *xe = base + lay.xe;
            const float *de = reinterpret_cast<const float *>(base + lay.de);
            const unsigned char *be = base + lay.be;
            const float *sB = reinterpret_cast<const float *>(base + lay.bc);
            const float *sC = reinterpret_cast<const float *>(base + lay.cs);
            const float4 *rowq = reinterpret_cast<const float4 *>(base + lay.rowq);
            float cv[kElemsPerThread];
            if (active) T::gather(sC, lane, cv);
            if (!fold) {
                // S_ckpt . C of this thread's rows (every lane of a row ends
                // with the sum) beside the B_j . C dots.
                float rsum[kReplayRows];
                if constexpr (SH == kShadowNone) {
                    if (active) {
#pragma unroll
                        for (int j = 0; j < kReplayRows; ++j) {
                            const int rr = slot_row + j * kReplaySlots;  // row within the tile
                            float sv[kElemsPerThread];
                            T::load_row_smem(tile + (rr < rows ? rr : 0) * N, lane, sv);
                            float acc = 0.f;
#pragma unroll
                            for (int i = 0; i < kElemsPerThread; ++i) acc = fmaf(sv[i], cv[i], acc);
                            rsum[j] = row_sum<L>(acc);
                        }
                    }
                } else if (active) {
                    // from the read copy: codes (times the row scale) or fp16
                    const unsigned char *copy = reinterpret_cast<const unsigned char *>(tile);
                    const float *rscale = reinterpret_cast<const float *>(copy + PS::kShadowScaleOffset);
#pragma unroll
                    for (int j = 0; j < kReplayRows; ++j) {
                        const int rr = slot_row + j * kReplaySlots;
                        const int rq = rr < rows ? rr : 0;
                        float sv[kElemsPerThread];
                        load_copy_row<TS, L>(copy, rq, lane, SH, sv);
                        float acc = 0.f;
#pragma unroll
                        for (int i = 0; i < kElemsPerThread; ++i) acc = fmaf(sv[i], cv[i], acc);
                        float rs = 1.f;
                        if constexpr (SH == kShadowE4M3) rs = rscale[rq];
                        if constexpr (SH == kShadowNVFP4)
                            rs = *reinterpret_cast<const float *>(copy + PS::kNvfp4RecOffset +
                                                                   rq * nvfp4_scale_words(N) * 4);
                        rsum[j] = row_sum<L>(acc) * rs;
                    }
                }
                entry_dots<N, kConsumers, IO>(c, be, sB, sC, dots, tid);
                named_barrier(1, kConsumers);
                if (active) {
                    // The walk of each row over entries c (the current token)
                    // down to 0, split in L contiguous parts, lane 0 the
                    // newest: each lane folds its part into {product of the
                    // decays, sum of the terms dt'_j x_j (B_j . C) weighted by
                    // the decays of the newer entries of the part}; the parts
                    // combine newest first, (w1, h1) then (w2, h2) giving
                    // (w1 w2, h1 + w1 h2).  The readout only produces y, so
                    // its decays take the fast exponential.
                    const int per = (c + L) / L;  // ceil((c + 1) / L)
                    const int hi = c - lane * per;
                    const int lo = hi - per + 1 > 0 ? hi - per + 1 : 0;
                    float w[kReplayRows], hs[kReplayRows];
                    float4 q[kReplayRows];
                    int rq[kReplayRows];
#pragma unroll
                    for (int j = 0; j < kReplayRows; ++j) {
                        const int rr = slot_row + j * kReplaySlots;
                        rq[j] = rr < rows ? rr : 0;
                        q[j] = rowq[rq[j]];
                        w[j] = 1.f;
                        hs[j] = 0.f;
                    }
                    int e = hi;
                    if (e == c) {
                        const float dc = dots[c];
#pragma unroll
                        for (int j = 0; j < kReplayRows; ++j) {
                            hs[j] = fmaf(q[j].y, dc, 0.f);
                            w[j] = q[j].x;
                        }
                        --e;
                    }
                    for (; e >= lo; --e) {
                        const float de_ = dots[e];
#pragma unroll
                        for (int j = 0; j < kReplayRows; ++j) {
                            const float d = de[e * kDtStride + rq[j]];
                            const float t = d * io_at<IO>(xe, e * x_stride<IO>() + rq[j]);
                            hs[j] = fmaf(w[j] * t, de_, hs[j]);
                            w[j] *= __expf(Ah * d);
                        }
                    }
#pragma unroll
                    for (int off = 1; off < L; off <<= 1) {
#pragma unroll
                        for (int j = 0; j < kReplayRows; ++j) {
                            const float w2 = __shfl_down_sync(0xffffffffu, w[j], off);
                            const float h2 = __shfl_down_sync(0xffffffffu, hs[j], off);
                            if ((lane & (2 * off - 1)) == 0) {
                                hs[j] = fmaf(w[j], h2, hs[j]);
                                w[j] *= w2;
                            }
                        }
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int j = 0; j < kReplayRows; ++j) {
                            const int rr = slot_row + j * kReplaySlots;
                            if (rr < rows)
                                store_small(p.y, cu.b * p.ys[0] + cu.h * p.ys[1] + (cu.row0 + rr) * p.ys[2], IO,
                                            output(fmaf(w[j], rsum[j], hs[j]), Dh, q[j].z, q[j].w));
                        }
                    }
                }
            } else {
                if (c > 0) {
                    entry_terms<kConsumers, IO>(c, rows, Ah, de, xe, rowa, rowb, tid);
                    named_barrier(1, kConsumers);
                }
                if (active) {
                    float bv[kElemsPerThread];
                    for (int j = 0; j < kReplayRows; ++j) {
                        const int rr = slot_row + j * kReplaySlots;
                        const bool live = rr < rows;
                        const int rq = live ? rr : 0;
                        float sv[kElemsPerThread];
                        if (seeded && live) {
                            T::load_row_smem(tile + rr * N, lane, sv);
                        } else {
#pragma unroll
                            for (int i = 0; i < kElemsPerThread; ++i) sv[i] = 0.f;
                        }
                        // The buffered steps in order, as the plain update made them ...
                        for (int e = 0; e < c; ++e) {
                            gather_entry<TS, L, IO>(be + e * N * io, lane, bv);
                            const float a = rowa[e * kTileRows + rq], dx = rowb[e * kTileRows + rq];
#pragma unroll
                            for (int i = 0; i < kElemsPerThread; ++i) sv[i] = fmaf(sv[i], a, dx * bv[i]);
                        }
                        // ... then the current token, whose state y is read from.
                        T::gather(sB, lane, bv);
                        const float4 q = rowq[rq];
                        const float sum = row_sum<L>(update_elems(sv, bv, cv, q.x, q.y));
                        if (live && lane == 0)
                            store_small(p.y, cu.b * p.ys[0] + cu.h * p.ys[1] + (cu.row0 + rr) * p.ys[2], IO,
                                        output(sum, Dh, q.z, q.w));
                        if (live && seeded) T::store_row_smem(tile + rr * N, lane, sv);
                        if constexpr (SH != kShadowNone) {
                            if (seeded)
                                write_copy_row<TS, L, SH>(
                                    p, (hd->slot * p.H + cu.h) * static_cast<int64_t>(p.P) + cu.row0 + rr, lane, live, sv);
                        }
                    }
                }
            }
        }
        if (stores) fence_proxy_async_smem();
        named_barrier(1, kConsumers);
        if (tid == 0) {
            if (stores) {
                unsigned char *dst = reinterpret_cast<unsigned char *>(
                    static_cast<TS *>(p.state) + ((hd->slot * p.H + cu.h) * static_cast<int64_t>(p.P) + cu.row0) * N);
                bulk_store(dst, base, static_cast<uint32_t>(cu.rows_here) * N * sizeof(TS));
                bulk_commit();
                if (S == 1) {
                    // One stage: the producer needs it back before the next unit.
                    bulk_wait_read<0>();
                    mbar_arrive(&empty[s]);
                } else {
                    // The previous store has had a unit's time to read its stage out.
                    if (pending >= 0) {
                        bulk_wait_read<1>();
                        mbar_arrive(&empty[pending]);
                    }
                    pending = s;
                }
            } else {
                if (pending >= 0) {
                    bulk_wait_read<0>();
                    mbar_arrive(&empty[pending]);
                    pending = -1;
                }
                mbar_arrive(&empty[s]);
            }
        }
    }
    if (tid == 0) bulk_wait_all();
    return k;
}

template <typename TS, int L, int IO, int SH>
__global__ void __launch_bounds__(ReplayPipe<TS, L, SH>::kThreads, ReplayPipe<TS, L, SH>::kMinCtas)
    ssu_replay_kernel(const KParams p, const ReplayLayout lay, int64_t units) {
    using PS = ReplayPipe<TS, L, SH>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *empty = full + lay.stages;
    RingExit *rx = reinterpret_cast<RingExit *>(smem + lay.exit);
    if (threadIdx.x == 0) {
        for (int s = 0; s < lay.stages; ++s) {
            mbar_init(&full[s], 32);
            mbar_init(&empty[s], 1);
        }
        ring_init(rx);
    }
    __syncthreads();
    const int warp = threadIdx.x / 32;
    int consumed = 0;
    if (warp >= PS::kConsumerWarps)
        replay_producer<TS, L, IO, SH>(p, lay, units, smem, full, empty, rx, warp - PS::kConsumerWarps);
    else
        consumed = replay_consumer<TS, L, IO, SH>(p, lay, units, smem, full, empty, rx);
    __syncthreads();
    if (threadIdx.x == 0) ring_drain(rx, full, lay.stages, consumed, p.wait_cycles, p.status);
}

// Dynamic shared memory the CTAs of one SM may take in all: the device's
// shared memory per SM less a 6 KB margin (222 KB of 228 KB on this part),
// and what one CTA may opt in to (cached per device).
static cudaError_t replay_smem_budget(int *per_sm, int *per_cta) {
    static std::atomic<int> cache_sm[64], cache_cta[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) dev = 0;
    int sm = cache_sm[dev].load(std::memory_order_relaxed), cta = cache_cta[dev].load(std::memory_order_relaxed);
    if (sm == 0 || cta == 0) {
        if ((e = cudaDeviceGetAttribute(&sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&cta, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return e;
        sm -= 6 * 1024;
        cache_sm[dev].store(sm, std::memory_order_relaxed);
        cache_cta[dev].store(cta, std::memory_order_relaxed);
    }
    *per_sm = sm;
    *per_cta = cta;
    return cudaSuccess;
}

// Number of SMs of the current device (cached per device).
static int replay_sm_count() {
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

// Once per device: opt in to the largest dynamic shared memory a CTA takes,
// and find how many CTAs of the kernel fit an SM by registers.
template <typename TS, int L, int IO, int SH>
static cudaError_t prepare_replay_kernel(int *reg_ctas) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        int per_sm = 0, per_cta = 0;
        if ((e = replay_smem_budget(&per_sm, &per_cta)) != cudaSuccess) return e;
        e = cudaFuncSetAttribute(ssu_replay_kernel<TS, L, IO, SH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 per_sm - 1024 < per_cta ? per_sm - 1024 : per_cta);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes a;
        e = cudaFuncGetAttributes(&a, ssu_replay_kernel<TS, L, IO, SH>);
        if (e != cudaSuccess) return e;
        const int regs = (a.numRegs + 7) / 8 * 8;  // allocated per thread in units of 8
        n = regs > 0 ? 65536 / (regs * ReplayPipe<TS, L, SH>::kThreads) : 1;
        if (n < 1) n = 1;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    *reg_ctas = n;
    return cudaSuccess;
}

template <typename TS, int L, int IO, int SH>
static cudaError_t launch_replay_t(const KParams &p, int64_t batch, cudaStream_t stream) {
    using PS = ReplayPipe<TS, L, SH>;
    int reg_ctas = 0;
    cudaError_t e = prepare_replay_kernel<TS, L, IO, SH>(&reg_ctas);
    if (e != cudaSuccess) return e;
    int per_sm = 0, per_cta = 0;
    if ((e = replay_smem_budget(&per_sm, &per_cta)) != cudaSuccess) return e;
    ReplayLayout lay;
    if (!lay.choose(PS::kTileBytes, PS::kN, p.rlen, IO == kF32 ? 4 : 2, per_sm, reg_ctas, PS::kProducerWarps) ||
        lay.bytes > per_cta)
        return cudaErrorInvalidConfiguration;
    const int64_t units = batch * p.H * p.ptiles;
    const int sms = replay_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int64_t slots_on_gpu = static_cast<int64_t>(sms) * lay.ctas;
    const int64_t grid = units < slots_on_gpu ? units : slots_on_gpu;
    ssu_replay_kernel<TS, L, IO, SH><<<static_cast<unsigned>(grid), PS::kThreads, lay.bytes, stream>>>(p, lay, units);
    return cudaGetLastError();
}

// The NVFP4 read copy needs a 16-element block to lie within one row's
// lanes (dstate 64 and up; the host rejects the rest).
template <typename TS, int LN, int IO>
static cudaError_t launch_replay_nvfp4(const KParams &p, int64_t batch, cudaStream_t stream) {
    if constexpr (LN % (16 / Tile<TS, LN>::kVec) == 0 && Tile<TS, LN>::kN >= 64)
        return launch_replay_t<TS, LN, IO, kShadowNVFP4>(p, batch, stream);
    else
        return cudaErrorInvalidValue;
}

template <typename TS, int IO>
static cudaError_t launch_replay_lanes(int lanes, const KParams &p, int64_t batch, cudaStream_t stream) {
    // one kernel per read-copy format: each carries only its own paths
    switch (lanes * 4 + p.shadow_fmt) {
#define SSU_REPLAY_CASE(LN)                                                                          \
    case LN * 4 + kShadowNone: return launch_replay_t<TS, LN, IO, kShadowNone>(p, batch, stream);   \
    case LN * 4 + kShadowF16: return launch_replay_t<TS, LN, IO, kShadowF16>(p, batch, stream);     \
    case LN * 4 + kShadowE4M3: return launch_replay_t<TS, LN, IO, kShadowE4M3>(p, batch, stream);   \
    case LN * 4 + kShadowNVFP4: return launch_replay_nvfp4<TS, LN, IO>(p, batch, stream);
        SSU_REPLAY_CASE(1)
        SSU_REPLAY_CASE(2)
        SSU_REPLAY_CASE(4)
        SSU_REPLAY_CASE(8)
        SSU_REPLAY_CASE(16)
#undef SSU_REPLAY_CASE
    }
    return cudaErrorInvalidValue;
}

// The replay launcher for operands of dtype IO (instantiated in one
// translation unit per IO).
template <int IO>
cudaError_t launch_replay_io(int state_dtype, int lanes, const KParams &p, int64_t batch, cudaStream_t stream) {
    switch (state_dtype) {
    case kF32: return launch_replay_lanes<float, IO>(lanes, p, batch, stream);
    case kF16: return launch_replay_lanes<__half, IO>(lanes, p, batch, stream);
    case kBF16: return launch_replay_lanes<__nv_bfloat16, IO>(lanes, p, batch, stream);
    }
    return cudaErrorInvalidValue;
}

extern template cudaError_t launch_replay_io<kF32>(int, int, const KParams &, int64_t, cudaStream_t);
extern template cudaError_t launch_replay_io<kF16>(int, int, const KParams &, int64_t, cudaStream_t);
extern template cudaError_t launch_replay_io<kBF16>(int, int, const KParams &, int64_t, cudaStream_t);

}  // namespace ssu
