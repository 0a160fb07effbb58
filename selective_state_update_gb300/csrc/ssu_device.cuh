// ssu_device.cuh -- device-side building blocks shared by the one-token and
// the packed kernel, so that a packed call whose sequences all have one token
// computes bit-for-bit what the one-token kernel computes.
//
// Thread layout of a work unit (one head, kTileRows dim rows, all of dstate):
//   L = dstate / 16 lanes cover one state row; the CTA has kRowSlots * L
//   threads; thread t serves row slot t / L and lane t % L, i.e. dim rows
//   slot, slot + kRowSlots, slot + 2 kRowSlots, slot + 3 kRowSlots of the
//   tile.  Within a row the thread owns the 16-byte chunks lane, lane + L,
//   lane + 2L, ... so each load/store instruction of a warp touches whole
//   128-byte lines.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "ssu_internal.h"

namespace ssu {

enum : int { kF32 = 0, kF16 = 1, kBF16 = 2 };  // ssu_dtype values

// ---------------------------------------------------------------------------
// Small operands (x, z, dt, B, C, y): dtype chosen at run time (uniform branch).
// ---------------------------------------------------------------------------
// Raw bits of element i of a small operand (32-bit types: the word; 16-bit
// types: the half-word).  Loads that are only converted later can all be in
// flight at once; converting right after each load would expose every
// load's latency in turn.
template <bool WIDE>
__device__ __forceinline__ uint32_t load_bits(const void *base, int64_t i) {
    if (WIDE) return __ldg(static_cast<const unsigned int *>(base) + i);
    return __ldg(static_cast<const unsigned short *>(base) + i);
}

__device__ __forceinline__ float to_float(float v) { return v; }
__device__ __forceinline__ float to_float(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }

// The low-precision read copy of a state row (article "ReplaySSM", section
// 低精度读写分离), E4M3 form: over the row's stored values, the dequantising
// scale amax / 448 and the quantising factor 448 / amax (both fp32, both 1
// for an all-zero row, the factor clamped to the largest finite float);
// code = E4M3(v * factor), the product in fp32, rounded to nearest even and
// clamped to +-448 (the conversion's saturate-to-finite mode).
__device__ __forceinline__ float shadow_scale_of(float amax) { return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f; }
__device__ __forceinline__ float shadow_factor_of(float amax) {
    return amax > 0.f ? fminf(__fdiv_rn(448.f, amax), 3.402823466e38f) : 1.f;
}
__device__ __forceinline__ unsigned char e4m3_code(float v) {
    return static_cast<unsigned char>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_value(unsigned int code) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code & 0xffu), __NV_E4M3)));
}

// NVFP4 form of the read copy: FP4 E2M1 codes, two a byte (the even element
// in the low nibble); per block of 16 elements an E4M3 scale code; per row an
// fp32 scale s = amax / (6 * 448), the row's record holding s and then the
// block codes, padded to a multiple of 16 bytes.  The block code is
// E4M3((block amax) / (6 s)) and an element's code E2M1(v / (block scale *
// s)), the quotients in fp32, both roundings to nearest even and saturating.
__host__ __device__ constexpr int nvfp4_scale_words(int n) { return (4 + n / 16 + 15) / 16 * 4; }
__device__ __forceinline__ float nvfp4_row_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 2688.f) : 1.f; }
__device__ __forceinline__ unsigned int nvfp4_block_code(float bmax, float s) {
    return e4m3_code(__fdiv_rn(bmax, __fmul_rn(6.f, s)));
}
// The byte of two E2M1 codes of a and b (a in the low nibble).
__device__ __forceinline__ unsigned int e2m1x2_code(float a, float b) {
    return __nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
}
// The two values of a byte of E2M1 codes (the low nibble first).
__device__ __forceinline__ float2 e2m1x2_values(unsigned int byte) {
    __half2_raw h = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte & 0xffu), __NV_E2M1);
    return __half22float2(__half2(h));
}
// Two values from two codes (the low byte first), one conversion.
__device__ __forceinline__ float2 e4m3x2_values(unsigned int codes) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes & 0xffffu), __NV_E4M3);
    return __half22float2(__half2(h));
}
// Two codes (a in the low byte) from two values, one conversion.
__device__ __forceinline__ unsigned int e4m3x2_codes(float a, float b) {
    return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}


__device__ __forceinline__ float bits_to_float(uint32_t v, int dtype) {
    if (dtype == kF32) return __uint_as_float(v);
    if (dtype == kBF16) return __uint_as_float(v << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v)));
}

__device__ __forceinline__ void store_small(void *base, int64_t i, int dtype, float v) {
    if (dtype == kF32) {
        static_cast<float *>(base)[i] = v;
    } else if (dtype == kBF16) {
        static_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half *>(base)[i] = __float2half_rn(v);
    }
}

__device__ __forceinline__ int64_t load_index(const void *base, int64_t i, int is_i64) {
    return is_i64 ? static_cast<int64_t>(__ldg(static_cast<const long long *>(base) + i))
                  : static_cast<int64_t>(__ldg(static_cast<const int *>(base) + i));
}

enum : int { kDevBadSlot = 0x1, kDevBadEntry = 0x2, kDevBadSeqlen = 0x4, kDevTimeout = 0x8, kDevBadCount = 0x10,
             kDevBadCopy = 0x20 };

__device__ __forceinline__ void flag(int32_t *status, int bit) {
    if (status != nullptr) atomicOr(status, bit);
}

// ---------------------------------------------------------------------------
// State chunks: 16 bytes of the pool <-> floats, rounded to nearest even.
// ---------------------------------------------------------------------------
template <typename TS>
struct StateChunk;

template <>
struct StateChunk<float> {
    static constexpr int kVec = 4;
    __device__ __forceinline__ static void unpack(const uint4 &u, float *v) {
        v[0] = __uint_as_float(u.x);
        v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z);
        v[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float *v) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
};

template <>
struct StateChunk<__half> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 &u, float *v) {
        const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 f = __half22float2(h);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
    __device__ __forceinline__ static uint4 pack(const float *v) {
        unsigned w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<unsigned *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct StateChunk<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ __forceinline__ static void unpack(const uint4 &u, float *v) {
        const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bf16 -> fp32 is a shift: exact.
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float *v) {
        unsigned w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<unsigned *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// ---------------------------------------------------------------------------
// Bulk asynchronous copy (TMA engine) of a contiguous state tile into shared
// memory, completed on an mbarrier.  Inline PTX for sm_90+ / sm_103a.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
    // Make the initialised barrier visible to the async proxy (TMA).
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once and expect `bytes` of transaction completions on this phase.
__device__ __forceinline__ void mbar_arrive_expect(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// global -> shared, `bytes` a multiple of 16, both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// shared -> global bulk copy (TMA engine), tracked in the issuing thread's
// bulk groups.  `bytes` a multiple of 16, both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_store(void *dst_gmem, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed (writes done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Barrier `id` over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier `id` over `nthreads` threads (a multiple of 32) that also returns
// whether any participant passed `v` true.
__device__ __forceinline__ bool barrier_or(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of `bar`; gives up after `limit` SM clock cycles
// (about a second at the default: a copy that never lands), or after 2^26
// polls, and returns false.
constexpr long long kWaitCycles = kDefaultWaitCycles;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) break;
    }
    return false;
}

// Exit of the ring kernels (one-token, packed, checkpoint + buffer).  Every
// wait is bounded.  When one gives up, its role sets `abort` and leaves; the
// producers stop filling stages once they see it.  All roles then meet at
// the CTA's last barrier, and one consumer thread waits (bounded) for every
// stage whose fill was issued but not consumed, so that no bulk copy still
// targets the CTA's shared memory when it retires.  `filled[s]` is the round
// of the last fill issued on stage s, plus one (0: none); fills of a stage
// come in order and a refill needs the previous round consumed, so at most
// one fill per stage is outstanding.
constexpr int kMaxRingStages = 8;
struct RingExit {
    int abort;
    int filled[kMaxRingStages];
};

__device__ __forceinline__ void ring_init(RingExit *r) {
    r->abort = 0;
    for (int s = 0; s < kMaxRingStages; ++s) r->filled[s] = 0;
}
__device__ __forceinline__ bool ring_aborted(const RingExit *r) {
    return *reinterpret_cast<const volatile int *>(&r->abort) != 0;
}
__device__ __forceinline__ void ring_abort(RingExit *r) { *reinterpret_cast<volatile int *>(&r->abort) = 1; }
// By the producer lane that issued the fill, after issuing its copies.
__device__ __forceinline__ void ring_note_fill(RingExit *r, int s, int round) {
    *reinterpret_cast<volatile int *>(&r->filled[s]) = round + 1;
}
// After the last barrier, by the consumer thread that counted `consumed`
// stages (the ring index of the first stage it did not consume).
__device__ __forceinline__ void ring_drain(const RingExit *r, uint64_t *full, int stages, long long consumed,
                                          long long limit, int32_t *status) {
    for (int s = 0; s < stages; ++s) {
        const int f = *reinterpret_cast<const volatile int *>(&r->filled[s]);
        if (f == 0) continue;
        const long long k = static_cast<long long>(f - 1) * stages + s;
        if (k >= consumed && !mbar_wait_bounded(&full[s], (f - 1) & 1, limit)) flag(status, kDevTimeout);
    }
}

// Streaming (evict-first) 16-byte accesses: each state byte is used once.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    return __ldcs(static_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
    __stcs(static_cast<uint4 *>(p), v);
}

// ---------------------------------------------------------------------------
// Per-thread view of a work unit.
// ---------------------------------------------------------------------------
template <typename TS, int L>
struct Tile {
    static constexpr int kVec = StateChunk<TS>::kVec;       // elements per 16-byte chunk
    static constexpr int kChunks = kElemsPerThread / kVec;   // chunks per thread per row
    static constexpr int kN = kElemsPerThread * L;           // dstate
    static constexpr int kThreads = kRowSlots * L;

    // Element offset (within a state row) of element i of this thread.
    __device__ __forceinline__ static int elem(int lane, int i) {
        return (lane + L * (i / kVec)) * kVec + (i % kVec);
    }

    // Load one row (16 elements) of this thread; row == nullptr gives zeros.
    __device__ __forceinline__ static void load_row(const TS *row, int lane, float *s) {
        if (row == nullptr) {
#pragma unroll
            for (int i = 0; i < kElemsPerThread; ++i) s[i] = 0.f;
            return;
        }
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
            uint4 u = ld_stream(row + (lane + L * k) * kVec);
            StateChunk<TS>::unpack(u, s + k * kVec);
        }
    }

    // Load one row (16 elements) of this thread from a tile in shared memory.
    __device__ __forceinline__ static void load_row_smem(const TS *row, int lane, float *s) {
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
            uint4 u = *reinterpret_cast<const uint4 *>(row + (lane + L * k) * kVec);
            StateChunk<TS>::unpack(u, s + k * kVec);
        }
    }

    // Store one row (16 elements) of this thread into a tile in shared memory.
    __device__ __forceinline__ static void store_row_smem(TS *row, int lane, const float *s) {
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
            *reinterpret_cast<uint4 *>(row + (lane + L * k) * kVec) = StateChunk<TS>::pack(s + k * kVec);
    }

    __device__ __forceinline__ static void store_row(TS *row, int lane, const float *s) {
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
            st_stream(row + (lane + L * k) * kVec, StateChunk<TS>::pack(s + k * kVec));
    }

    // This thread's 16 values of a dstate vector staged in shared memory.
    __device__ __forceinline__ static void gather(const float *smem, int lane, float *v) {
#pragma unroll
        for (int k = 0; k < kChunks; ++k) {
#pragma unroll
            for (int q = 0; q < kVec / 4; ++q) {
                float4 f = *reinterpret_cast<const float4 *>(smem + (lane + L * k) * kVec + 4 * q);
                v[k * kVec + 4 * q + 0] = f.x;
                v[k * kVec + 4 * q + 1] = f.y;
                v[k * kVec + 4 * q + 2] = f.z;
                v[k * kVec + 4 * q + 3] = f.w;
            }
        }
    }
};

// Sum over the L lanes of a row (lanes of a row are consecutive lane ids).
template <int L>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// dt' for one (row, head, dim row): dt (+ bias), softplus if asked.
// softplus(v) = log(1 + e^v) in the form max(v, 0) + log1p(e^-|v|).
__device__ __forceinline__ float step_size(float dt, float bias, int softplus) {
    float v = dt + bias;
    if (softplus) v = fmaxf(v, 0.f) + log1pf(expf(-fabsf(v)));
    return v;
}

// One token applied to this thread's 16 elements of one state row:
// S = S * dA + (dt' x) * B, and the partial sum of S * C over those elements
// (four interleaved partial sums, so that the dependent chain is four FMAs
// long instead of sixteen; every kernel uses this order).
__device__ __forceinline__ float update_elems(float *s, const float *b, const float *c, float dA,
                                              float dtx) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kElemsPerThread; ++i) {
        s[i] = fmaf(s[i], dA, dtx * b[i]);
        acc[i % 4] = fmaf(s[i], c[i], acc[i % 4]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// y = (sum + D x) * gate, gate = silu(z) (or 1 without z).
__device__ __forceinline__ float output(float sum, float Dh, float x, float gate) {
    return fmaf(Dh, x, sum) * gate;
}

// Inputs of one (row, head, dim row): dt, x, z (z = 0 without a gate).
struct RowInputs {
    float dt, x, z;
};

// The processed step dt' and the decay exp(A dt').  Not inlined, so that the
// kernels, and a later fold of a buffered step, all get the same bits.
static __device__ __noinline__ float processed_step(float dt, float bias, int softplus) {
    return step_size(dt, bias, softplus);
}
// exp(A dt') with the product rounded on its own (never fused into an
// FMA), so that an inlined copy gives the bits of the call.
__device__ __forceinline__ float decay_inline(float Ah, float d) { return expf(__fmul_rn(Ah, d)); }
static __device__ __noinline__ float decay(float Ah, float d) { return decay_inline(Ah, d); }

// The factor y is multiplied by: silu(z) = z / (1 + e^-z) with a z input,
// 1 without.  Not inlined, like the two above.
static __device__ __noinline__ float silu_gate(float z, int has_z) { return has_z ? z / (1.f + expf(-z)) : 1.f; }

// Per-row scalars {dA, dt' x, x, gate}, from the calls above only: every
// kernel gets exactly the same instructions, hence the same bits.
static __device__ __noinline__ float4 row_scalars(RowInputs in, float Ah, float bias, int softplus, int has_z) {
    const float d = processed_step(in.dt, bias, softplus);
    const float gate = silu_gate(in.z, has_z);
    return make_float4(decay(Ah, d), d * in.x, in.x, gate);
}

// (sequence, head, dim tile) of a work unit of the one-token style kernels.
struct UnitCoords {
    int64_t b;
    int h, g, row0, rows_here;
};

// Walks this CTA's units u = blockIdx.x + k * gridDim.x as (sequence, head,
// dim tile) with additions and carries only: no 64-bit division per unit.
struct UnitWalker {
    int pt, h;          // current dim tile and head
    int64_t b;          // current sequence
    int d_pt, d_h;      // the stride gridDim.x as (tiles, heads, sequences)
    int64_t d_b;

    __device__ __forceinline__ UnitWalker(const KParams &p, int64_t u, int64_t step) {
        pt = static_cast<int>(u % p.ptiles);
        h = static_cast<int>((u / p.ptiles) % p.H);
        b = u / (static_cast<int64_t>(p.ptiles) * p.H);
        d_pt = static_cast<int>(step % p.ptiles);
        d_h = static_cast<int>((step / p.ptiles) % p.H);
        d_b = step / (static_cast<int64_t>(p.ptiles) * p.H);
    }
    __device__ __forceinline__ void advance(const KParams &p) {
        pt += d_pt;
        int carry = 0;
        if (pt >= p.ptiles) {
            pt -= p.ptiles;
            carry = 1;
        }
        h += d_h + carry;
        carry = 0;
        if (h >= p.H) {
            h -= p.H;
            carry = 1;
        }
        b += d_b + carry;
    }
    __device__ __forceinline__ UnitCoords coords(const KParams &p) const {
        UnitCoords c;
        c.b = b;
        c.h = h;
        c.g = h / p.heads_per_group;
        c.row0 = pt * kTileRows;
        c.rows_here = min(kTileRows, p.P - c.row0);
        return c;
    }
};

// Slot at entry (b, t) of table `t`, or `fallback` without a table.  Returns
// false (and flags) when the entry lies outside the table.
__device__ __forceinline__ bool table_slot(const KParams &p, const SlotTab &t, int64_t b,
                                           int64_t step, int64_t row_start, int64_t fallback,
                                           int64_t *slot) {
    if (t.entries == nullptr) {
        *slot = fallback;
        return true;
    }
    const int64_t e = t.per_row ? row_start + step : b * t.s0 + step * t.s1;
    if (e < 0 || e >= t.extent) {
        flag(p.status, kDevBadEntry);
        return false;
    }
    *slot = load_index(t.entries, e, t.is_i64);
    return true;
}

// A slot is usable if it is the pad id or inside the pool.
__device__ __forceinline__ bool slot_ok(const KParams &p, int64_t s) {
    if (s == p.pad || (s >= 0 && s < p.slots)) return true;
    flag(p.status, kDevBadSlot);
    return false;
}

// Everything the producer needs from global memory for one unit, loaded into
// registers one unit ahead so that the loads are in flight while the producer
// stages the previous unit or waits for a free stage.  The loads are issued
// as raw bits, back to back, and converted only when the unit is staged.
template <typename TS, int L>
struct UnitOperands {
    static constexpr int kN = Tile<TS, L>::kN;
    static constexpr int kPerB = (kN + 31) / 32;
    static constexpr int kPerRow = (kTileRows + 31) / 32;
    UnitCoords c;
    int64_t rs, ws;  // lane 0: raw slots (valid when entries_ok)
    bool entries_ok;
    uint32_t b[kPerB], cc[kPerB];
    uint32_t dt[kPerRow], x[kPerRow], z[kPerRow];
    float Ah, bias, Dh;

    template <bool WIO, bool WDT>
    __device__ __forceinline__ void load_operands(const KParams &p, int lane) {
        const int64_t bo = c.b * p.Bs[0] + c.g * p.Bs[1];
        const int64_t co = c.b * p.Cs[0] + c.g * p.Cs[1];
#pragma unroll
        for (int i = 0; i < kPerB; ++i) {
            const int n = lane + 32 * i;
            if (n < kN) {
                b[i] = load_bits<WIO>(p.B, bo + n * p.Bs[2]);
                cc[i] = load_bits<WIO>(p.C, co + n * p.Cs[2]);
            }
        }
#pragma unroll
        for (int i = 0; i < kPerRow; ++i) {
            const int pr = c.row0 + lane + 32 * i;
            if (lane + 32 * i < c.rows_here) {
                dt[i] = load_bits<WDT>(p.dt, c.b * p.dts[0] + c.h * p.dts[1] + pr * p.dts[2]);
                x[i] = load_bits<WIO>(p.x, c.b * p.xs[0] + c.h * p.xs[1] + pr * p.xs[2]);
                z[i] = p.z ? load_bits<WIO>(p.z, c.b * p.zs[0] + c.h * p.zs[1] + pr * p.zs[2]) : 0u;
            }
        }
    }

    __device__ __forceinline__ void load(const KParams &p, const UnitCoords &cu, int lane) {
        c = cu;
        entries_ok = true;
        rs = ws = 0;
        if (lane == 0) {
            entries_ok = table_slot(p, p.rd, c.b, 0, c.b, c.b, &rs);
            if (p.wr.entries != nullptr)
                entries_ok = table_slot(p, p.wr, c.b, 0, c.b, c.b, &ws) && entries_ok;
        }
        const bool wio = p.io_dtype == kF32, wdt = p.dt_dtype == kF32;
        if (wio) {
            if (wdt) load_operands<true, true>(p, lane);
            else load_operands<true, false>(p, lane);
        } else {
            if (wdt) load_operands<false, true>(p, lane);
            else load_operands<false, false>(p, lane);
        }
        Ah = __ldg(p.A + c.h);
        bias = p.dt_bias ? __ldg(p.dt_bias + c.h) : 0.f;
        Dh = p.D ? __ldg(p.D + c.h) : 0.f;
    }
};

}  // namespace ssu
