// ssd_tc.cu -- bf16 chunked SSD forward on tcgen05 tensor cores (sm_103a).
//
// Work unit: one chunk of Q tokens of one "head block" -- the 128 / headdim
// heads (2 for headdim 64, 1 for headdim 128) whose headdim rows fill the
// 128 lanes of a tensor-memory accumulator.  All heads of a block share one
// B/C group.  Operands arrive by TMA in 128-byte-swizzled 64-column slabs;
// accumulators live in TMEM; one thread issues the MMAs.  The chunk algebra is
// written out in ssd_internal.cuh.
//
// chunk_state_tc:  S_c[(h,p), n] = sum_j w_{h,j} x_j[h,p] B_j[n],
//                  w_{h,j} = exp(cs_last - cs_j) dt_j           (M=128, N=dstate, K=chunk)
//                  w*x is fed as two bf16 terms (hi + lo): a single rounding of it
//                  costs up to ~2.4% of RMS(final_state) on short sequences.  32-token
//                  slabs, three in flight; S_c leaves by TMA through swizzled fp32 boxes.
// (state_pass_hilo, in ssd_simt.cu, turns S_c into the entry states h_c, in place, as
//  bf16 hi + lo terms per 64-wide slice of the state dimension.)
// chunk_out_tc:    persistent; per tile = (128 rows i0 .. i0+127 of a chunk, head block),
//                  columns j < i0 + 128:
//                  G    = C_i B_j^T                              (M=128, N=i0+128, K=dstate)
//                  Yoff = C_i (h_hi + h_lo)^T  (both heads)       (M=128, N=128,    K=dstate)
//                         the carried state can be ~10x larger than y (an init state), and a
//                         single bf16 rounding of it alone costs ~2% of RMS(y)
//                  S_h  = G o exp(cs_i - cs_j) dt_j [j <= i]  as hi + lo bf16 in shared memory
//                         (rank-one decays when the chunk's decay range allows)
//                  Ydiag_h = S_hi x_h + S_lo x_h                  (M=128, N=headdim, K=i0+128)
//                  y = Ydiag + exp(cs_i) Yoff + D x
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "ssd_internal.cuh"
#include "ssd_ptx.cuh"

namespace ssd {
namespace {

using namespace ptx;

constexpr int kThreads = 128;      // chunk_state_tc: the working threads (warps 0-3) ...
constexpr int kStThreads = 160;    // ... and warp 4, which issues its loads, MMAs and stores
constexpr int kBoxRows = 128;           // tokens per TMA box
constexpr int kBoxBytes = 64 * 2 * kBoxRows;  // 64 bf16 columns x 128 rows = 16 KiB
// chunk_state_tc goes through the chunk in 32-token slabs, a ring of three in flight: its
// shared memory (97 KiB at dstate 256) leaves room for two CTAs per SM
constexpr int kStRows = 32;
constexpr int kStBytes = 64 * 2 * kStRows;    // 64 bf16 columns x 32 rows = 4 KiB
constexpr int kStStages = 3;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void set_error(const Problem &pr, unsigned int flag)
{
    if (pr.err_word) atomicOr(pr.err_word, flag);
}

// Barrier of threads 0-127 of a larger block, while its other warps work on.
__device__ __forceinline__ void sync128() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// Inclusive prefix sum of 256 values held two per thread (thread t holds
// values 2t and 2t+1) across threads 0-127.  warp_tot: 4 floats.
__device__ __forceinline__ void scan_128x2(float &v0, float &v1, float *warp_tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float own = v0 + v1;
    float s = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += t;
    }
    if (lane == 31) warp_tot[warp] = s;
    sync128();
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off += warp_tot[w];
    sync128();
    v0 = off + (s - own) + v0;
    v1 = v0 + v1;
}

// Segment sums of one chunk for the heads h0 .. h0+nh-1: cs[hh][j] (in-chunk
// inclusive prefix of dt*A*scale, 0 beyond the chunk) and dtv[hh][j] (0 beyond
// the chunk).  Rows are 256 floats apart.  Returns nothing; ends synchronised.
__device__ __forceinline__ void segsum(const Problem &pr, int b, int h0, int nh, int t0, int len, float scale,
                                       float *cs, float *dtv, float *warp_tot)
{
    const int t = threadIdx.x;
    const int j0 = 2 * t, j1 = 2 * t + 1;
    // every head's loads first (nh <= 2), so that their latencies overlap
    float d0[2], d1[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const size_t o = ((size_t)b * pr.seqlen + t0) * pr.nheads + h0 + hh;
        d0[hh] = hh < nh && j0 < len ? __ldg(pr.dt + o + (size_t)j0 * pr.nheads) : 0.f;
        d1[hh] = hh < nh && j1 < len ? __ldg(pr.dt + o + (size_t)j1 * pr.nheads) : 0.f;
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        if (hh >= nh) break;  // block-uniform
        const int h = h0 + hh;
        const float a = __ldg(pr.A + h) * scale;
        float v0 = d0[hh] * a, v1 = d1[hh] * a;
        scan_128x2(v0, v1, warp_tot);
        cs[hh * 256 + j0] = v0;
        cs[hh * 256 + j1] = v1;
        if (pr.dtin) {  // input scale
            dtv[hh * 256 + j0] = j0 < len ? __ldg(pr.dtin + ((size_t)b * pr.seqlen + t0 + j0) * pr.nheads + h) : 0.f;
            dtv[hh * 256 + j1] = j1 < len ? __ldg(pr.dtin + ((size_t)b * pr.seqlen + t0 + j1) * pr.nheads + h) : 0.f;
        } else {
            dtv[hh * 256 + j0] = d0[hh];
            dtv[hh * 256 + j1] = d1[hh];
        }
    }
    sync128();
}

// The chunk's cumulative decays in two steps, so that the loads of dt can be issued
// long before the scan needs them: seg_load reads thread t's token of each head
// (nh <= 2); seg_scan writes the scaled inclusive prefix sums of dt * A into cs and
// the per-token dt (dt_in when the caller passed one) into dtv.
struct SegRegs {
    float d[2], din[2];
};

__device__ __forceinline__ SegRegs seg_load(const Problem &pr, int b, int h0, int nh, int t0, int len)
{
    SegRegs r;
    const int t = threadIdx.x;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const bool on = hh < nh && t < len;
        const size_t o = ((size_t)b * pr.seqlen + t0 + t) * pr.nheads + h0 + hh;
        r.d[hh] = on ? __ldg(pr.dt + o) : 0.f;
        r.din[hh] = on && pr.dtin ? __ldg(pr.dtin + o) : 0.f;  // no use of a loaded value here
    }
    return r;
}

// Barrier of the 256 threads (warps 0-7) of a larger block, while its other warps work on.
__device__ __forceinline__ void sync256() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Inclusive scan of one value per thread over threads 0-255 (named barrier 1).
__device__ __forceinline__ float scan256_named(float v, float *warp_tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    sync256();
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off += warp_tot[w];
    sync256();  // warp_tot is reused by the next call
    return v + off;
}

// Called by threads 0-255 only.
__device__ __forceinline__ void seg_scan(const Problem &pr, const SegRegs &r, int h0, int nh, float scale, float *cs,
                                         float *dtv, float *warp_tot)
{
    const int t = threadIdx.x;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        if (hh < nh) {  // block-uniform
            const float a = __ldg(pr.A + h0 + hh) * scale;
            cs[hh * 256 + t] = scan256_named(r.d[hh] * a, warp_tot);
            dtv[hh * 256 + t] = pr.dtin ? r.din[hh] : r.d[hh];
        }
    }
    sync256();
}

// Pack 8 floats into 8 bf16 (one 16-byte chunk).
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

// Byte offset of logical 16-B chunk q (0..7) of row r in a 128-B-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int q) { return (uint32_t)r * 128u + (uint32_t)((q ^ (r & 7)) << 4); }

// ---------------------------------------------------------------------------
// chunk state
// ---------------------------------------------------------------------------

template <int NS>
__global__ void __launch_bounds__(kStThreads, 1)
    chunk_state_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bmap,
                   const __grid_constant__ CUtensorMap smap, Problem pr, Workspace ws)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma[kStStages], bar_mma[kStStages], bar_built[kStStages];
    __shared__ uint32_t tmem_slot;
    __shared__ float warp_tot[4];
    __shared__ float cs[2 * 256], dtv[2 * 256];
    __shared__ int s_fail;

    const int hb = blockIdx.y;
    const ChunkRef ref = chunk_ref(pr, blockIdx.x, blockIdx.z);
    const int P = pr.headdim, HB = 128 / P, H = pr.nheads;
    const int h0 = hb * HB, g = h0 / (H / pr.ngroups);
    const int b = ref.tb, t0 = ref.t0, len = ref.len;  // b: batch row of the token tensors
    const int nbox = (pr.chunk + kStRows - 1) / kStRows;  // 32-token slabs along K
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // slab kh in stage kh % 3: w*x as hi and lo bf16 terms (2 MN blocks of 64 (h,p)
    // columns each) and B (NS/64 MN blocks of 64 n columns)
    uint8_t *base = align1024(smem_raw);
    constexpr int kStage = (4 + NS / 64) * kStBytes;
    auto xs_of = [&](int st) { return base + st * kStage; };                 // x, then hi(w*x) in place
    auto xl_of = [&](int st) { return base + st * kStage + 2 * kStBytes; };  // lo(w*x)
    auto bs_of = [&](int st) { return base + st * kStage + 4 * kStBytes; };  // B

    if (tid == 0) {
        for (int k = 0; k < kStStages; ++k) {
            mbar_init(&bar_tma[k], 1);
            mbar_init(&bar_mma[k], 1);
            mbar_init(&bar_built[k], kThreads);  // the working threads, once per slab
        }
        mbar_fence_init();
        s_fail = 0;
    }
    if (warp == 0) tmem_alloc(&tmem_slot, NS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    auto issue_loads = [&](int kh) {
        const int st = kh % kStStages;
        uint64_t *bar = &bar_tma[st];
        mbar_expect_tx(bar, (uint32_t)((2 + NS / 64) * kStBytes));
        for (int k = 0; k < 2; ++k)
            tma_load_3d(xs_of(st) + k * kStBytes, &xmap, bar, hb * 128 + 64 * k, t0 + kh * kStRows, b);
        for (int s = 0; s < NS / 64; ++s)
            tma_load_3d(bs_of(st) + s * kStBytes, &bmap, bar, g * NS + 64 * s, t0 + kh * kStRows, b);
    };
    bool ok;
    if (warp == 4) {
        // warp 4: the loads of the first three slabs, then per slab the MMAs once every
        // working thread has built it, and the loads of slab kh + 2 into the stage of slab
        // kh - 1 once that slab's MMAs are done
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            tma_prefetch_desc(&bmap);
            tma_prefetch_desc(&smap);
            for (int kh = 0; kh < kStStages && kh < nbox; ++kh) issue_loads(kh);
            bool good = true;
            for (int kh = 0; kh < nbox && good; ++kh) {
                const int st = kh % kStStages;
                if (!mbar_wait(&bar_built[st], (uint32_t)(kh / kStStages) & 1u)) {
                    good = false;
                    break;
                }
                tc_fence_after();
                constexpr uint32_t idesc = idesc_bf16(128, NS, 1, 1);
                const uint32_t xa = smem_u32(xs_of(st)), xla = smem_u32(xl_of(st)), ba = smem_u32(bs_of(st));
                for (int ks = 0; ks < kStRows / 16; ++ks) {
                    const uint64_t bd = sdesc_sw128(ba + ks * 2048, kStBytes, 1024);
                    mma_bf16(tmem, sdesc_sw128(xa + ks * 2048, kStBytes, 1024), bd, idesc, (kh | ks) != 0);
                    mma_bf16(tmem, sdesc_sw128(xla + ks * 2048, kStBytes, 1024), bd, idesc, 1);
                }
                mma_commit(&bar_mma[st]);
                if (kh >= 1 && kh + 2 < nbox) {
                    if (!mbar_wait(&bar_mma[(kh - 1) % kStStages], (uint32_t)((kh - 1) / kStStages) & 1u)) {
                        good = false;
                        break;
                    }
                    issue_loads(kh + 2);
                }
            }
            // every slab's MMAs done (this thread has seen slab nbox - 4's complete, so the
            // parity wait cannot mistake the barrier's previous phase)
            if (good && !mbar_wait(&bar_mma[(nbox - 1) % kStStages], (uint32_t)((nbox - 1) / kStStages) & 1u))
                good = false;
            if (!good) s_fail = 1;
        }
        __syncwarp();
    } else {
        // segment sums and decay-to-chunk-end weights (natural-log domain, accurate exp)
        segsum(pr, b, h0, HB, t0, len, 1.f, cs, dtv, warp_tot);
        float *wts = cs;  // overwrite cs with w after reading cs_last
        const float cl0 = cs[len - 1], cl1 = HB > 1 ? cs[256 + len - 1] : 0.f;
        sync128();
        for (int e = tid; e < HB * 256; e += kThreads) {
            const int j = e & 255;
            wts[e] = j >= len ? 0.f : pr.adjoint_states ? expf(cs[e]) : expf((e < 256 ? cl0 : cl1) - cs[e]) * dtv[e];
        }
        if (tid < HB && !pr.adjoint_states) ws.decay[state_slot(pr, ref, h0 + tid)] = expf(tid == 0 ? cl0 : cl1);
        sync128();

        // slab kh: wait for its loads, build w*x, arrive; the stage is rewritten only by the
        // loads of slab kh + 3, which warp 4 issues after slab kh's MMAs are done
        for (int kh = 0; kh < nbox; ++kh) {
            const int st = kh % kStStages;
            uint8_t *xs = xs_of(st), *xl = xl_of(st);
            const bool landed = mbar_wait(&bar_tma[st], (uint32_t)(kh / kStStages) & 1u);
            if (!landed) s_fail = 1;
            // w*x -> hi (in place) + lo; one 16-B chunk = 8 columns of one token row
            for (int q = tid; q < 2 * kStRows * 8 && landed; q += kThreads) {
                const int k = q / (kStRows * 8), row = (q / 8) % kStRows;
                const float w = wts[(P == 64 ? k : 0) * 256 + kh * kStRows + row];
                uint4 *ptr = reinterpret_cast<uint4 *>(xs) + q;
                uint4 v = *ptr;
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
                float f[8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 t = __bfloat1622float2(h2[u]);
                    f[2 * u] = t.x * w;
                    f[2 * u + 1] = t.y * w;
                }
                const uint4 hi = pack8(f);
                const __nv_bfloat162 *hh2 = reinterpret_cast<const __nv_bfloat162 *>(&hi);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 t = __bfloat1622float2(hh2[u]);
                    f[2 * u] -= t.x;
                    f[2 * u + 1] -= t.y;
                }
                *ptr = hi;
                reinterpret_cast<uint4 *>(xl)[q] = pack8(f);
            }
            fence_async_smem();  // the slab, written here, is read by the tensor cores
            mbar_arrive(&bar_built[st]);
        }
    }
    __syncthreads();  // warp 4 has seen the last MMAs complete
    tc_fence_after();
    ok = !s_fail;
    // S_c out: 32 state columns at a time into a [128 rows][32] fp32 box with the 128-byte
    // swizzle (double-buffered over the dead stages), each head's P rows stored by
    // TMA as one box of the [state rows][NS] view of the workspace
    if (ok) {  // warps 0-3 stage the rows (their TMEM lanes), lane 0 of warp 4 stores them
        const int m = warp * 32 + lane;
        const bool issuer = warp == 4 && lane == 0;
#pragma unroll 1
        for (int c0 = 0; c0 < NS; c0 += 32) {
            uint8_t *buf = base + ((c0 / 32) & 1) * 16384;  // [128 rows][32] fp32, over the dead stages
            if (c0 >= 64) {  // the store of two slabs ago must be done reading this buffer
                if (issuer) bulk_wait_read_1();
                __syncthreads();
            }
            if (warp < 4) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4 *>(buf + sw128(m, q)) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                fence_async_smem();
            }
            __syncthreads();
            if (issuer) {
                for (int hh = 0; hh < HB; ++hh)
                    tma_store_3d(&smap, buf + hh * P * 128, c0, (int)(state_slot(pr, ref, h0 + hh) * P), 0);
                bulk_commit();
            }
        }
        if (issuer) bulk_wait_read_all();
    } else if (tid == 0) {
        set_error(pr, kDevErrTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, NS);
}

// ---------------------------------------------------------------------------
// chunk output
// ---------------------------------------------------------------------------

// One phase-1 stage (the C | B | h_hi | h_lo slabs of one 64-wide slice of the state
// dimension): 64 KiB when the tile spans 128 columns, 80 KiB when it spans 256.  Two
// stages alternate.  Once the slices are done, the x tile takes the first 64 KiB and
// the masked S tiles (hi and lo terms) the next 128 KiB.
__host__ __device__ constexpr int stage_bytes(int jmax) { return jmax > 128 ? 80 * 1024 : 64 * 1024; }

// chunk_out_tc: warps w and w + 4 (w < 4) share TMEM lanes 32 w .. 32 w + 31, scan the
// decays while the slices are multiplied, then build S and run the epilogue; warp 8 issues
// every MMA and warp 9 every load of the slices, so that no building warp waits on either
constexpr int kOutThreads = 320;

template <int NS>
__global__ void __launch_bounds__(kOutThreads, 1)
    chunk_out_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bmap,
                 const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap ymap,
                 const __grid_constant__ CUtensorMap smap, Problem pr, Workspace ws)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma[2], bar_mma[2], bar_x, bar_mm2[2], bar_built[2];
    __shared__ uint32_t tmem_slot;
    __shared__ float warp_tot[8];
    __shared__ __align__(16) float cs[2 * 256];
    __shared__ __align__(16) float dtv[2 * 256];  // read as float4 in phase 2
    __shared__ float s_mn[2][8], s_mx[2][8];
    __shared__ int s_fail, s_next;

    const int ntile = pr.chunk <= kBoxRows ? 1 : 2;
    const int P = pr.headdim, HB = 128 / P, H = pr.nheads, L = pr.seqlen;
    const int nhb = H / HB;
    const int ncx = pr.chunks ? pr.total_chunks : pr.nchunks;
    const int ntiles = nhb * ntile * ncx * (pr.chunks ? 1 : pr.batch);
    // TMEM: G (jn columns), Ydiag and Yoff (128 each); one CTA per SM (its shared memory)
    const uint32_t tcols = 512;
    const uint32_t col_g = 0, col_yd = 256, col_yo = 384;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;  // TMEM lanes 32 quarter ..; half of the columns

    uint8_t *base = align1024(smem_raw);
    const int jmax = pr.chunk <= kBoxRows ? kBoxRows : 2 * kBoxRows;
    constexpr int nsl = NS / 64;                  // 64-wide slices of the state dimension
    // stage k: C (128 x 128 B) | B (jn x 128 B) | h_hi | h_lo (128 x 128 B each); slice s
    // uses stage (s + nsl) & 1, so that the last slice is in stage 1 and stage 0 is free
    // for the x tile once slice nsl - 2 (if any) is multiplied
    auto stage = [&](int sl) { return base + ((sl + nsl) & 1) * stage_bytes(jmax); };
    auto bar_of = [&](uint64_t *bars, int sl) { return &bars[(sl + nsl) & 1]; };
    uint8_t *xs = base;                           // x: 2 MN blocks, each jn x 128 B (<= 64 KiB)
    uint8_t *r1 = base + 65536;                   // S tiles (hi, lo) of a pass's heads: 128 KiB

    if (tid == 0) {
        mbar_init(&bar_tma[0], 1);
        mbar_init(&bar_tma[1], 1);
        mbar_init(&bar_mma[0], 1);
        mbar_init(&bar_mma[1], 1);
        mbar_init(&bar_x, 1);
        mbar_init(&bar_mm2[0], 1);
        mbar_init(&bar_mm2[1], 1);
        mbar_init(&bar_built[0], 256);  // every building thread, once per S chunk
        mbar_init(&bar_built[1], 256);
        mbar_fence_init();
        s_fail = 0;
    }
    if (warp == 0) tmem_alloc(&tmem_slot, tcols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    // Persistent: one CTA per SM takes tiles by ticket, head block fastest, so that the
    // head blocks of one chunk tile follow each other and share C and B in L2.  Every
    // mbarrier completes a known number of times per tile; the counts so far give the
    // parity each wait needs.
    if (warp == 9 && lane == 0) {
        tma_prefetch_desc(&smap);
        tma_prefetch_desc(&cmap);
        tma_prefetch_desc(&bmap);
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&ymap);
        s_next = (int)atomicAdd(ws.ticket, 1u);  // the first tile; warp 9 takes each next one early
    }
    uint32_t n_st0 = 0, n_st1 = 0, n_x = 0, n_s0 = 0, n_s1 = 0;
    for (;;) {
        tc_fence_before();
        __syncthreads();  // the previous tile is done with TMEM and shared memory
        tc_fence_after();
        const int tk = s_next;
        if (tk >= ntiles || s_fail) break;  // block-uniform
        const int hb = tk % nhb, it = (tk / nhb) % ntile, cxz = tk / (nhb * ntile);
        const ChunkRef ref = chunk_ref(pr, cxz % ncx, cxz / ncx);
        const int h0 = hb * HB, g = h0 / (H / pr.ngroups);
        const int b = ref.tb, t0 = ref.t0, len = ref.len;  // b: batch row of the token tensors
        const int i0 = it * kBoxRows;
        if (i0 >= len) {  // tile beyond the end of a partial last chunk (block-uniform)
            __syncthreads();  // every thread has read s_next
            if (warp == 9 && lane == 0) s_next = (int)atomicAdd(ws.ticket, 1u);
            continue;
        }
        const int jn = i0 + kBoxRows;                 // columns j in [0, jn)
        const int nbj = jn / kBoxRows;                // 128-row boxes along j
        // parity of the wait for slice s on its stage's barriers, for S chunk kc on its buffer's
        auto par_s = [&](int sl) { return (((sl + nsl) & 1 ? n_st1 : n_st0) + (uint32_t)(sl >> 1)) & 1u; };
        auto par_k = [&](int kc) { return ((kc & 1 ? n_s1 : n_s0) + (uint32_t)(kc >> 1)) & 1u; };

        // TMA issue (lane 0 of warp 9; lane 0 of warp 8 issues the MMAs).  A stage takes
        // slice sl of C_i and B_j and of each head's entry state
        // h_c, whose hi and lo bf16 terms the state pass laid out per slice (a [P][64] box of
        // each at columns 128 sl and 128 sl + 64 of the slot's [P][2 NS] bf16 rows).
        auto issue_stage = [&](int sl) {
            uint8_t *st = stage(sl);
            uint64_t *bar = bar_of(bar_tma, sl);
            mbar_expect_tx(bar, (uint32_t)((1 + nbj) * kBoxBytes + 2 * kBoxBytes));
            tma_load_3d(st, &cmap, bar, g * NS + 64 * sl, t0 + i0, b);
            for (int r = 0; r < nbj; ++r)
                tma_load_3d(st + kBoxBytes + r * kBoxBytes, &bmap, bar, g * NS + 64 * sl, t0 + r * kBoxRows, b);
            uint8_t *h_sl = st + kBoxBytes + jn * 128, *l_sl = h_sl + kBoxBytes;
            for (int hh = 0; hh < HB; ++hh) {
                const int row = (int)(state_slot(pr, ref, h0 + hh) * P);
                tma_load_3d(h_sl + hh * P * 128, &smap, bar, 128 * sl, row, 0);
                tma_load_3d(l_sl + hh * P * 128, &smap, bar, 128 * sl + 64, row, 0);
            }
        };
        auto issue_x = [&]() {  // the x rows of the whole tile span, both 64-column blocks
            mbar_expect_tx(&bar_x, (uint32_t)(2 * nbj * kBoxBytes));
            for (int k = 0; k < 2; ++k)
                for (int r = 0; r < nbj; ++r)
                    tma_load_3d(xs + k * jn * 128 + r * kBoxBytes, &xmap, &bar_x, hb * 128 + 64 * k, t0 + r * kBoxRows,
                                b);
        };
        if (warp == 9 && lane == 0) {
            issue_stage(0);
            if (nsl > 1)
                issue_stage(1);
            else
                issue_x();  // stage 0 is not used by the one slice
            // the rest of the chunk's entry states (one P x NS block of hi / lo pairs per head,
            // from DRAM) into L2, so that the later slice loads find them there
            for (int hh = 0; hh < HB; ++hh)
                bulk_prefetch_l2(ws.states + state_slot(pr, ref, h0 + hh) * (size_t)P * NS, (uint32_t)(P * NS * sizeof(float)));
        }
        // ---- phase 1: G = C_i B^T and Yoff = C_i (h_hi + h_lo)^T over the 64-wide slices of
        // the state dimension, two stages in flight: slice s + 1 lands while slice s is
        // multiplied.  Meanwhile warps 0-7 scan the decays.
        constexpr float kFactorSpan = 160.f;  // log2 units (see below)
        float rowf[2] = {1.f, 1.f};
        bool factored = false;
        if (warp < 8) {
            const SegRegs seg = seg_load(pr, b, h0, HB, t0, len);
            seg_scan(pr, seg, h0, HB, kLog2e, cs, dtv, warp_tot);  // log2 domain: decays via ex2

            // The decays exp2(cs_i - cs_j) in rank-one form, exp2(cs_i - ref) exp2(ref - cs_j)
            // with ref the midpoint of each head's cs range over the chunk, whenever that range is
            // at most kFactorSpan (every factor then within 2^(+-kFactorSpan / 2) of 1): one exp
            // per row and per column instead of one per element of S.  The column factors, times
            // dt_j, replace dtv and go into S; the row factor multiplies row i of S x in the
            // epilogue.  A wider range keeps the exp per element (and a row factor of 1).
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const bool on = hh < HB && tid < len;
                const float cv = cs[hh * 256 + tid];
                float mn = on ? cv : 3.0e38f, mx = on ? cv : -3.0e38f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                }
                if (lane == 0) {
                    s_mn[hh][warp] = mn;
                    s_mx[hh][warp] = mx;
                }
            }
            sync256();
            float ref[2];
            factored = true;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float mn = s_mn[hh][0], mx = s_mx[hh][0];
#pragma unroll
                for (int w = 1; w < 8; ++w) {
                    mn = fminf(mn, s_mn[hh][w]);
                    mx = fmaxf(mx, s_mx[hh][w]);
                }
                ref[hh] = 0.5f * (mn + mx);
                if (hh < HB && !(mx - mn <= kFactorSpan)) factored = false;  // uniform over warps 0-7
            }
            if (factored) {
                const int ir = i0 + (warp & 3) * 32 + lane;  // this thread's accumulator row in phase 2
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (hh < HB) {
                        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(rowf[hh]) : "f"(cs[hh * 256 + (ir < 256 ? ir : 255)] - ref[hh]));
                        float c;
                        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(c) : "f"(ref[hh] - cs[hh * 256 + tid]));
                        dtv[hh * 256 + tid] = tid < len ? c * dtv[hh * 256 + tid] : 0.f;
                    }
                }
            }
        } else if (warp == 8) {
            if (lane == 0) {
                bool good = true;
                for (int s = 0; s < nsl && good; ++s) {
                    uint8_t *c_sl = stage(s), *b_sl = c_sl + kBoxBytes, *h_sl = b_sl + jn * 128, *l_sl = h_sl + kBoxBytes;
                    if (!mbar_wait(bar_of(bar_tma, s), par_s(s))) {
                        good = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t id_g = idesc_bf16(128, jn, 0, 0);
                    constexpr uint32_t id_o = idesc_bf16(128, 128, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(smem_u32(c_sl) + kk * 32, 16, 1024);
                        mma_bf16(tmem + col_g, ad, sdesc_sw128(smem_u32(b_sl) + kk * 32, 16, 1024), id_g,
                                 (s | kk) != 0);
                        mma_bf16(tmem + col_yo, ad, sdesc_sw128(smem_u32(h_sl) + kk * 32, 16, 1024), id_o,
                                 (s | kk) != 0);
                        mma_bf16(tmem + col_yo, ad, sdesc_sw128(smem_u32(l_sl) + kk * 32, 16, 1024), id_o, 1);
                    }
                    mma_commit(bar_of(bar_mma, s));
                }
                if (!good) s_fail = 1;
            }
            __syncwarp();
        } else {  // warp 9
            if (lane == 0) {
                // the other stage is free once slice s - 1's MMAs are done: slice s + 1 goes
                // there, or, after the last slice, the x tile (stage 0)
                bool good = true;
                for (int s = 1; s < nsl && good; ++s) {
                    if (!mbar_wait(bar_of(bar_mma, s - 1), par_s(s - 1))) {
                        good = false;
                        break;
                    }
                    if (s + 1 < nsl)
                        issue_stage(s + 1);
                    else
                        issue_x();
                }
                if (!good) s_fail = 1;
            }
            __syncwarp();
        }
        // every slice's MMAs done (the last commit covers all earlier MMAs of warp 8).  Warp 8
        // alone waits: it has seen slice nsl - 3's MMAs complete, so the parity wait cannot
        // mistake the barrier's previous phase for this one; the others learn it at the barrier.
        if (warp == 8 && !mbar_wait(bar_of(bar_mma, nsl - 1), par_s(nsl - 1))) s_fail = 1;
        __syncthreads();  // also publishes cs and the column factors
        tc_fence_after();
        bool ok = !s_fail;

        // ---- phase 2: S_h = G o decay o dt (causal) as hi + lo bf16 terms (a single rounding of
        // S costs up to 2^-9 |y_i| where one term dominates a row, i.e. under strong decay, when
        // |y| reaches ~10x its RMS); Ydiag_h = S_hi x_h + S_lo x_h.  S goes in K-chunks of 128
        // columns (head-major), double-buffered in 64 KiB (hi, then lo): chunk k + 1 is built
        // while chunk k is multiplied.
        const int i = quarter * 32 + lane;    // accumulator row of this thread
        const int ia = i0 + i;                // row within the chunk
        const bool row_ok = ia < len;
        const int nhalf = jn / 128;           // K-chunks per head
        const int nkc = ok ? HB * nhalf : 0;  // block-uniform
        if (warp < 8) {
            for (int kc = 0; kc < nkc; ++kc) {
                const int hh = kc / nhalf, jh = kc % nhalf;
                uint8_t *buf = r1 + (kc & 1) * 65536;
                // the buffer was last read by the MMAs of chunk kc - 2
                if (kc >= 2 && !mbar_wait(&bar_mm2[kc & 1], par_k(kc - 2))) s_fail = 1;
                const float *csh = cs + hh * 256, *dth = dtv + hh * 256;
                const float ci = csh[ia < 256 ? ia : 255];
                for (int lb = half; lb < 4; lb += 2) {  // 32-column blocks lb of the chunk: warps 0-3 even, 4-7 odd
                    const int j0 = 128 * jh + 32 * lb;
                    uint8_t *st = buf + (lb / 2) * kBoxBytes;
                    const int cq = (lb & 1) * 4;          // first 16-byte column of the block in its 64-column box
                    if (j0 > i0 + quarter * 32 + 31) {  // whole warp above the diagonal: zeros
                        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            *reinterpret_cast<uint4 *>(st + sw128(i, cq + u)) = z;
                            *reinterpret_cast<uint4 *>(st + 32768 + sw128(i, cq + u)) = z;
                        }
                        continue;
                    }
                    float gv[32];
                    tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + col_g + j0, gv);
                    // cs and dt (or the column factors) of the block's 32 columns as float4s
                    float sv[32];
                    // every row of the warp in the chunk and past the block's last column: no mask
                    const bool full = j0 + 31 <= i0 + quarter * 32 && i0 + quarter * 32 + 31 < len;
                    if (factored && full) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 f4 = reinterpret_cast<const float4 *>(dth + j0)[q];
                            sv[4 * q] = gv[4 * q] * f4.x;
                            sv[4 * q + 1] = gv[4 * q + 1] * f4.y;
                            sv[4 * q + 2] = gv[4 * q + 2] * f4.z;
                            sv[4 * q + 3] = gv[4 * q + 3] * f4.w;
                        }
                    } else if (factored) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 f4 = reinterpret_cast<const float4 *>(dth + j0)[q];
                            const float fj[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const int k = 4 * q + v, j = j0 + k;
                                // masked entries (j > row) are discarded, whatever the product is
                                sv[k] = (row_ok && j <= ia) ? gv[k] * fj[v] : 0.f;
                            }
                        }
                    } else {
                        // the decays by the hardware base-2 exponential (ex2.approx, relative error ~2^-22)
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 c4 = reinterpret_cast<const float4 *>(csh + j0)[q];
                            const float4 d4 = reinterpret_cast<const float4 *>(dth + j0)[q];
                            const float cj[4] = {c4.x, c4.y, c4.z, c4.w}, dj[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const int k = 4 * q + v, j = j0 + k;
                                float e;  // masked entries (j > row) are discarded below, whatever e is
                                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(ci - cj[v]));
                                sv[k] = (row_ok && j <= ia) ? gv[k] * e * dj[v] : 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 hi = pack8(sv + 8 * u);
                        const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&hi);
                        float r[8];
#pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) {
                            const float2 t = __bfloat1622float2(h2[e2]);
                            r[2 * e2] = sv[8 * u + 2 * e2] - t.x;
                            r[2 * e2 + 1] = sv[8 * u + 2 * e2 + 1] - t.y;
                        }
                        *reinterpret_cast<uint4 *>(st + sw128(i, cq + u)) = hi;
                        *reinterpret_cast<uint4 *>(st + 32768 + sw128(i, cq + u)) = pack8(r);
                    }
                }
                fence_async_smem();  // the S chunk, written here, is read by the tensor cores
                mbar_arrive(&bar_built[kc & 1]);
            }
        } else if (warp == 8 && lane == 0) {  // the MMAs of each S chunk once every building thread has arrived
            bool good = true;
            for (int kc = 0; kc < nkc && good; ++kc) {
                const int hh = kc / nhalf, jh = kc % nhalf;
                if (!mbar_wait(&bar_built[kc & 1], par_k(kc)) || (kc == 0 && !mbar_wait(&bar_x, n_x & 1u))) {
                    good = false;
                    break;
                }
                tc_fence_after();
                const uint32_t id_d = idesc_bf16(128, P, 0, 1);  // one head's headdim columns
                const uint32_t s_addr = smem_u32(r1 + (kc & 1) * 65536);
                const uint32_t x_addr = smem_u32(xs) + (P == 64 ? hh : 0) * jn * 128;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t so = (ks / 4) * kBoxBytes + (ks % 4) * 32;
                    const uint64_t bd = sdesc_sw128(x_addr + (8 * jh + ks) * 2048, jn * 128, 1024);
                    mma_bf16(tmem + col_yd + hh * P, sdesc_sw128(s_addr + so, 16, 1024), bd, id_d, (jh | ks) != 0);
                    mma_bf16(tmem + col_yd + hh * P, sdesc_sw128(s_addr + 32768 + so, 16, 1024), bd, id_d, 1);
                }
                mma_commit(&bar_mm2[kc & 1]);
            }
            if (!good) s_fail = 1;
        } else if (warp == 9 && lane == 0) {
            // idle here: take the next tile's ticket and bring its entry states and x rows
            // into L2, so that its first slices do not wait on DRAM
            const int tn = (int)atomicAdd(ws.ticket, 1u);
            s_next = tn;
            if (tn < ntiles) {
                const int hbn = tn % nhb, itn = (tn / nhb) % ntile, czn = tn / (nhb * ntile);
                const ChunkRef rn = chunk_ref(pr, czn % ncx, czn / ncx);
                if (itn * kBoxRows < rn.len) {
                    for (int hh = 0; hh < HB; ++hh)
                        bulk_prefetch_l2(ws.states + state_slot(pr, rn, hbn * HB + hh) * (size_t)P * NS,
                                         (uint32_t)(P * NS * sizeof(float)));
                    for (int k = 0; k < 2; ++k)
                        for (int r = 0; r <= itn; ++r)
                            tma_prefetch_l2_3d(&xmap, hbn * 128 + 64 * k, rn.t0 + r * kBoxRows, rn.tb);
                }
            }
        }
        __syncwarp();
        // every chunk's MMAs done (the last commit covers the earlier ones); warps 0-8 have seen
        // chunk nkc - 3's complete, warp 9 takes it from the barrier
        if (nkc > 0 && warp < 9 && !mbar_wait(&bar_mm2[(nkc - 1) & 1], par_k(nkc - 1))) s_fail = 1;
        __syncthreads();
        ok = !s_fail;
        tc_fence_after();

        // ---- phase 3: y = Ydiag + exp(cs_i) Yoff + D x, staged over this tile's x rows and
        // stored by TMA when the tile's 128 rows all belong to the chunk (the batch layout
        // with chunks of 128 or 256 tokens; rows past the sequence end are clipped by the
        // tensor map), else stored row by row
        const bool tma_out = !pr.chunks && (pr.chunk == kBoxRows || pr.chunk == 2 * kBoxRows);
        if (ok && !mbar_wait(&bar_x, n_x & 1u)) ok = false;  // x tile (already complete) visible to every thread
        if (ok && warp < 8) {
            const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
            for (int hh = 0; hh < HB; ++hh) {
                const int h = h0 + hh;
                const float e = exp2f(cs[hh * 256 + (ia < 256 ? ia : 255)]);
                const float rf = hh == 0 ? rowf[0] : rowf[1];  // 1 unless the decays are factored
                const float Dh = pr.D ? __ldg(pr.D + h) : 0.f;
                __nv_bfloat16 *yrow = static_cast<__nv_bfloat16 *>(pr.y) + (((size_t)b * L + t0 + ia) * H + h) * P;
                for (int p0 = half * (P / 2); p0 < (half + 1) * (P / 2); p0 += 32) {
                    float yd[32], yo[32];
                    tmem_ld32(tmem + lane_base + col_yd + hh * P + p0, yd);
                    tmem_ld32(tmem + lane_base + col_yo + hh * P + p0, yo);
                    if (row_ok || tma_out) {
                        const int col = hh * P + p0;            // column within the 128-wide x tile
                        uint8_t *xrow = xs + (col / 64) * jn * 128;
                        uint4 ov[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint4 xv = *reinterpret_cast<const uint4 *>(xrow + sw128(ia, (col % 64) / 8 + u));
                            const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
                            float out[8];
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const float2 xf = __bfloat1622float2(x2[v]);
                                const int k = 8 * u + 2 * v;
                                out[2 * v] = fmaf(rf, yd[k], fmaf(e, yo[k], Dh * xf.x));
                                out[2 * v + 1] = fmaf(rf, yd[k + 1], fmaf(e, yo[k + 1], Dh * xf.y));
                            }
                            ov[u] = pack8(out);
                        }
                        if (tma_out) {
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                *reinterpret_cast<uint4 *>(xrow + sw128(ia, (col % 64) / 8 + u)) = ov[u];
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(yrow + p0);
#pragma unroll
                            for (int u = 0; u < 4; ++u) dst[u] = ov[u];
                        }
                    }
                }
            }
        } else if (!ok && tid == 0) {
            set_error(pr, kDevErrTimeout);
        }
        if (tma_out) {
            fence_async_smem();
            __syncthreads();
            if (ok && tid == 0) {  // the tile's rows i0 .. i0 + 127 of both 64-column blocks
                for (int k = 0; k < 2; ++k)
                    tma_store_3d(&ymap, xs + k * jn * 128 + i0 * 128, hb * 128 + 64 * k, t0 + i0, b);
                bulk_commit();
                bulk_wait_read_all();
            }
        }
        // completions of this tile on each barrier
#pragma unroll
        for (int sl = 0; sl < nsl; ++sl) {
            if ((sl + nsl) & 1)
                ++n_st1;
            else
                ++n_st0;
        }
        ++n_x;
        n_s0 += (uint32_t)(nkc + 1) / 2;
        n_s1 += (uint32_t)nkc / 2;
    }  // tiles
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, tcols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [batch][seqlen][width] bf16 tensor viewed as 3-D, boxes of 64 columns x 128 tokens.
cudaError_t make_map(CUtensorMap *map, const void *ptr, int width, int seqlen, int batch)
{
    return cached_tensor_map(map, ptr, true, width, seqlen, batch, 64, kBoxRows, true);
}

size_t state_smem(const Problem &pr)
{
    return 1024 + std::max<size_t>((size_t)kStStages * (4 + pr.dstate / 64) * kStBytes, 2 * 16384);
}

size_t out_smem(const Problem &pr)
{
    const int jmax = pr.chunk <= kBoxRows ? kBoxRows : 2 * kBoxRows;
    // two stages of the slices; after them x (64 KiB at most) and 128 KiB of S tiles
    return 1024 + std::max<size_t>(2 * (size_t)stage_bytes(jmax), 65536 + 131072);
}

template <int NS>
cudaError_t launch_tc(const Problem &pr, const Workspace &ws, cudaStream_t s, int phase)
{
    CUtensorMap xmap, bmap, cmap;
    cudaError_t e;
    const int HB = 128 / pr.headdim;
    // packed sequences: one batch row of seqlen tokens, one CTA (row) per chunk-table entry
    const int mb = pr.chunks ? 1 : pr.batch;
    const int ncx = pr.chunks ? pr.total_chunks : pr.nchunks;
    if (phase == 0) {
        if ((e = cached_tensor_map(&xmap, pr.x, true, pr.nheads * pr.headdim, pr.seqlen, mb, 64, kStRows, true)) !=
            cudaSuccess)
            return e;
        if ((e = cached_tensor_map(&bmap, pr.B, true, pr.ngroups * pr.dstate, pr.seqlen, mb, 64, kStRows, true)) !=
            cudaSuccess)
            return e;
        // the chunk states as [state rows = slots x headdim][NS] fp32, boxes of headdim rows x 32
        CUtensorMap smap;
        const size_t slots = pr.chunks ? (size_t)pr.nheads * pr.total_chunks : (size_t)pr.batch * pr.nheads * pr.nchunks;
        if (slots * pr.headdim > (size_t)INT32_MAX) return cudaErrorInvalidValue;  // box row coordinates are 32-bit
        if ((e = cached_tensor_map(&smap, ws.states, false, NS, (int)(slots * pr.headdim), 1, 32, pr.headdim, true)) !=
            cudaSuccess)
            return e;
        const size_t smem = state_smem(pr);
        if ((e = ensure_smem_limit(reinterpret_cast<const void *>(chunk_state_tc<NS>), smem)) != cudaSuccess) return e;
        const dim3 grid(ncx, pr.nheads / HB, mb);
        profile_kernel_begin(s);
        chunk_state_tc<NS><<<grid, kStThreads, smem, s>>>(xmap, bmap, smap, pr, ws);
        profile_kernel_end(s);
    } else {
        if ((e = make_map(&xmap, pr.x, pr.nheads * pr.headdim, pr.seqlen, mb)) != cudaSuccess) return e;
        if ((e = make_map(&bmap, pr.B, pr.ngroups * pr.dstate, pr.seqlen, mb)) != cudaSuccess) return e;
        if ((e = make_map(&cmap, pr.C, pr.ngroups * pr.dstate, pr.seqlen, mb)) != cudaSuccess) return e;
        CUtensorMap ymap, smap;
        if ((e = make_map(&ymap, pr.y, pr.nheads * pr.headdim, pr.seqlen, mb)) != cudaSuccess) return e;
        // the entry states h_c as [state rows = slots x headdim][2 NS] bf16 (hi and lo terms per
        // 64-wide slice, as the state pass writes them), boxes of headdim rows x 64
        const size_t slots = pr.chunks ? (size_t)pr.nheads * pr.total_chunks : (size_t)pr.batch * pr.nheads * pr.nchunks;
        if (slots * pr.headdim > (size_t)INT32_MAX) return cudaErrorInvalidValue;  // box row coordinates are 32-bit
        if ((e = cached_tensor_map(&smap, ws.states, true, 2 * NS, (int)(slots * pr.headdim), 1, 64, pr.headdim,
                                   true)) != cudaSuccess)
            return e;
        const size_t smem = out_smem(pr);
        if ((e = ensure_smem_limit(reinterpret_cast<const void *>(chunk_out_tc<NS>), smem)) != cudaSuccess) return e;
        // persistent: one CTA per SM, tiles by ticket (the counter is zeroed per launch)
        const int ntile = pr.chunk <= kBoxRows ? 1 : 2;
        const long long tiles = (long long)ncx * ntile * (pr.nheads / HB) * mb;
        if (tiles > INT32_MAX) return cudaErrorInvalidValue;
        int sms = 148;
        if ((e = sm_count(&sms)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(ws.ticket, 0, sizeof(uint32_t), s)) != cudaSuccess) return e;
        const unsigned grid = (unsigned)std::min<long long>(tiles, sms);
        profile_kernel_begin(s);
        chunk_out_tc<NS><<<grid, kOutThreads, smem, s>>>(xmap, bmap, cmap, ymap, smap, pr, ws);
        profile_kernel_end(s);
    }
    return cudaGetLastError();
}

cudaError_t dispatch(const Problem &pr, const Workspace &ws, cudaStream_t s, int phase)
{
    switch (pr.dstate) {
    case 64: return launch_tc<64>(pr, ws, s, phase);
    case 128: return launch_tc<128>(pr, ws, s, phase);
    case 256: return launch_tc<256>(pr, ws, s, phase);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return encode_fn(); }

bool tc_supported(const Problem &pr)
{
    if (pr.dtype != SSD_DTYPE_BF16) return false;
    if (pr.headdim != 64 && pr.headdim != 128) return false;
    if (pr.dstate != 64 && pr.dstate != 128 && pr.dstate != 256) return false;
    if (pr.chunk > 2 * kBoxRows) return false;
    const int HB = 128 / pr.headdim;
    if (pr.nheads % HB != 0 || (pr.nheads / pr.ngroups) % HB != 0) return false;
    return true;
}

cudaError_t launch_chunk_state_tc(const Problem &pr, const Workspace &ws, cudaStream_t s)
{
    return dispatch(pr, ws, s, 0);
}

cudaError_t launch_chunk_out_tc(const Problem &pr, const Workspace &ws, cudaStream_t s)
{
    return dispatch(pr, ws, s, 1);
}

}  // namespace ssd
