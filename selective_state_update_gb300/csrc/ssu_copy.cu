// ssu_copy.cu -- batched state copies with memmove semantics.
//
// Digest of vLLM PR #50729, section 实现拆解 (items 1-4): speculative decoding
// shifts and moves slot state inside one buffer, so a copy's source and
// destination can overlap; a parallel memcpy then lets one lane overwrite
// bytes another lane has not read yet.  A copy must behave like memmove (the
// destination receives the source bytes as they were before the copy), and
// the price of that ordering is paid only by copies that really overlap
// (item 2, "快速路径与重叠路径分离"; item 4, the left-overlap test that
// upgrades memcpy to memmove).
//
// Copy i of a batch is one ssu_copy descriptor {src, dst, bytes} in device
// memory.  The grid is (tile slots, copies): copies that do not overlap
// themselves are cut into kTile-byte tiles copied independently by all tile
// slots (16-byte vector loads, all of a thread's loads in flight before its
// stores, when both addresses are 16-byte aligned; 4-byte or byte accesses
// otherwise).  A copy that overlaps itself is moved by its first CTA alone,
// through shared memory, one kStage-byte piece at a time in the order that
// never overwrites a byte before it has been read: ascending when the
// destination lies below the source, descending when above.  Within a piece
// every byte is read before any is written; a piece's writes reach only bytes
// already read (its own piece and the pieces before it in that order).
#include <cstdint>

#include "ssu_device.cuh"

namespace ssu {

struct CopyDesc {
    uint64_t src, dst, bytes;
};

constexpr int kCopyThreads = 256;
constexpr int kCopyVec = 16;                                  // uint4 per thread and tile
constexpr uint64_t kTile = uint64_t(kCopyThreads) * kCopyVec * 16;  // 64 KiB
constexpr int kStage = 32 * 1024;                             // bytes per ordered piece

// Bytes [lo, hi) of a non-overlapping copy, 16-byte aligned addresses.
__device__ __forceinline__ void copy_tile_vec(const unsigned char *src, unsigned char *dst, uint64_t lo,
                                              uint64_t hi) {
    const uint64_t n16 = (hi - lo) / 16;
    const uint4 *s = reinterpret_cast<const uint4 *>(src + lo);
    uint4 *d = reinterpret_cast<uint4 *>(dst + lo);
    if (n16 == kTile / 16) {
        uint4 v[kCopyVec];
#pragma unroll
        for (int k = 0; k < kCopyVec; ++k) v[k] = __ldcs(s + threadIdx.x + k * kCopyThreads);
#pragma unroll
        for (int k = 0; k < kCopyVec; ++k) __stcs(d + threadIdx.x + k * kCopyThreads, v[k]);
    } else {
        for (uint64_t k = threadIdx.x; k < n16; k += kCopyThreads) __stcs(d + k, __ldcs(s + k));
    }
    for (uint64_t k = lo + n16 * 16 + threadIdx.x; k < hi; k += kCopyThreads) dst[k] = src[k];
}

// Bytes [lo, hi) of a non-overlapping copy, any alignment.
__device__ __forceinline__ void copy_tile_any(const unsigned char *src, unsigned char *dst, uint64_t lo,
                                              uint64_t hi, bool words) {
    if (words) {  // both addresses and the tile start 4-byte aligned
        const uint64_t n4 = (hi - lo) / 4;
        const uint32_t *s = reinterpret_cast<const uint32_t *>(src + lo);
        uint32_t *d = reinterpret_cast<uint32_t *>(dst + lo);
        for (uint64_t k = threadIdx.x; k < n4; k += kCopyThreads) d[k] = s[k];
        lo += n4 * 4;
    }
    for (uint64_t k = lo + threadIdx.x; k < hi; k += kCopyThreads) dst[k] = src[k];
}

// A copy that overlaps itself: one CTA, pieces in the safe order.
__device__ void copy_ordered(const unsigned char *src, unsigned char *dst, uint64_t bytes, unsigned char *stage) {
    const bool ascending = dst < src;
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    const uint64_t pieces = (bytes + kStage - 1) / kStage;
    for (uint64_t i = 0; i < pieces; ++i) {
        const uint64_t piece = ascending ? i : pieces - 1 - i;
        const uint64_t lo = piece * kStage;
        const uint64_t n = bytes - lo < uint64_t(kStage) ? bytes - lo : uint64_t(kStage);
        const uint64_t n16 = vec ? n / 16 : 0;
        for (uint64_t k = threadIdx.x; k < n16; k += kCopyThreads)
            reinterpret_cast<uint4 *>(stage)[k] = reinterpret_cast<const uint4 *>(src + lo)[k];
        for (uint64_t k = n16 * 16 + threadIdx.x; k < n; k += kCopyThreads) stage[k] = src[lo + k];
        __syncthreads();  // the whole piece is read ...
        for (uint64_t k = threadIdx.x; k < n16; k += kCopyThreads)
            reinterpret_cast<uint4 *>(dst + lo)[k] = reinterpret_cast<const uint4 *>(stage)[k];
        for (uint64_t k = n16 * 16 + threadIdx.x; k < n; k += kCopyThreads) dst[lo + k] = stage[k];
        __syncthreads();  // ... and written before the next one is read
    }
}

__global__ void __launch_bounds__(kCopyThreads)
    ssu_copy_kernel(const CopyDesc *copies, int64_t n, uint64_t max_bytes, int32_t *status) {
    __shared__ __align__(16) unsigned char stage[kStage];
    for (int64_t i = blockIdx.y; i < n; i += gridDim.y) {
        const CopyDesc c{__ldg(&copies[i].src), __ldg(&copies[i].dst), __ldg(&copies[i].bytes)};
        if (c.bytes == 0 || c.src == c.dst) continue;
        if (c.bytes > max_bytes) {  // larger than the caller's bound: skipped
            if (blockIdx.x == 0 && threadIdx.x == 0) flag(status, kDevBadCopy);
            continue;
        }
        const unsigned char *src = reinterpret_cast<const unsigned char *>(c.src);
        unsigned char *dst = reinterpret_cast<unsigned char *>(c.dst);
        const bool overlap = c.dst < c.src + c.bytes && c.src < c.dst + c.bytes;
        if (overlap) {
            if (blockIdx.x == 0) copy_ordered(src, dst, c.bytes, stage);
            continue;
        }
        const bool vec = ((c.src | c.dst) & 15) == 0;
        const bool words = ((c.src | c.dst) & 3) == 0;
        for (uint64_t lo = uint64_t(blockIdx.x) * kTile; lo < c.bytes; lo += uint64_t(gridDim.x) * kTile) {
            const uint64_t hi = c.bytes - lo < kTile ? c.bytes : lo + kTile;
            if (vec)
                copy_tile_vec(src, dst, lo, hi);
            else
                copy_tile_any(src, dst, lo, hi, words);
        }
    }
}

cudaError_t launch_copy(const void *copies, int64_t n, uint64_t max_bytes, int32_t *status, cudaStream_t stream) {
    uint64_t tiles = (max_bytes + kTile - 1) / kTile;
    if (tiles > 4096) tiles = 4096;  // each CTA then loops over several tiles
    const int64_t ys = n < 65535 ? n : 65535;
    ssu_copy_kernel<<<dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(ys)), kCopyThreads, 0, stream>>>(
        static_cast<const CopyDesc *>(copies), n, max_bytes, status);
    return cudaGetLastError();
}

}  // namespace ssu
