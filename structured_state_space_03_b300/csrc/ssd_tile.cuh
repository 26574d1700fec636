// ssd_tile.cuh -- small device helpers of the fused tcgen05 kernels: the
// 128-byte-swizzled tile addressing of TMA / tcgen05 operands, bf16 packing and
// the hi + lo split, named barriers, gpu-scope flag accesses.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ssd {
namespace tile {

constexpr int kRows = 128;              // tokens per tile, TMEM lanes
constexpr int kSlab = 64 * 2 * kRows;   // 64 bf16 columns x 128 rows = 16 KiB

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Byte offset of the 16-byte chunk q (0..7) of row r in a 128-byte-swizzled slab
// (rows of 128 bytes, chunk index XOR-ed with the row's low three bits).
__device__ __forceinline__ uint32_t sw128(int r, int q) { return (uint32_t)r * 128u + (uint32_t)((q ^ (r & 7)) << 4); }

__device__ __forceinline__ uint4 pack8(const float *f)
{
    uint4 u;
    __nv_bfloat162 t;
    t = __floats2bfloat162_rn(f[0], f[1]);
    u.x = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2bfloat162_rn(f[2], f[3]);
    u.y = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2bfloat162_rn(f[4], f[5]);
    u.z = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2bfloat162_rn(f[6], f[7]);
    u.w = *reinterpret_cast<uint32_t *>(&t);
    return u;
}

// hi = bf16(f), lo = bf16(f - hi), 8 values (round to nearest even both times)
__device__ __forceinline__ void split8(const float *f, uint4 &hi, uint4 &lo)
{
    hi = pack8(f);
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&hi);
    float r[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 t = __bfloat1622float2(h2[u]);
        r[2 * u] = f[2 * u] - t.x;
        r[2 * u + 1] = f[2 * u + 1] - t.y;
    }
    lo = pack8(r);
}

// Named barrier `id` over `n` threads.
__device__ __forceinline__ void named_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier over `n` threads that also returns whether any of them passed `pred`.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Release store of a publication flag: ordered after every write this thread
// observed, including those of the threads it met at a barrier just before.
__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

}  // namespace tile
}  // namespace ssd
