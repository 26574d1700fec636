// ssd_fused.cu -- single-kernel bf16 SSD forward on tcgen05 (sm_103a) for
// chunk <= 128, headdim 64/128, dstate 64/128.
//
// A unit is (chunk c, batch b, head block hb), a head block being the
// 128/headdim heads whose (head, headdim) rows fill the 128 TMEM lanes.  x, B
// and C of the chunk are read from HBM once and y is written once; the
// chunk-to-chunk recurrence h_{c+1} = a_c h_c + S_c is resolved between units
// by a decoupled look-back over states published in the workspace.  dstate 128
// runs one CTA (256 threads) per unit (ssd_fused_tc, described here); dstate
// 64 runs the persistent ssd_fused_pipe_tc further down, one CTA per SM with two
// units in flight, on the same arithmetic.
//
// Inside the chunk the decay exp(cs_i - cs_j) is rank one per head:
//   exp(cs_i - cs_j) = r_i v_j,  r_i = exp(cs_i - ref),  v_j = exp(ref - cs_j)
// with ref the midpoint of the chunk's cs range, so both factors stay within
// e^(+-60) whenever the range ("span") is at most 120.  Then (ssd_internal.cuh)
//   S_c          = e^(cs_last - ref) (v o dt o x)^T B
//   y_i          = r_i [ sum_{j<=i} (C_i . B_j) wx_j  +  e^ref C_i . h_c ]  +  D x_i,
//   wx_j         = v_j dt_j x_j
// and the masked matrix tril(C B^T) no longer depends on the head: one bf16
// copy of it serves every head of the block, and a single accumulator holds
// both matrix products.  wx (as hi + lo bf16 terms) is the operand of both the
// chunk-state and the diagonal-block GEMM.  Steps:
//
//   1. TMA x, B, C; segment sums, span, ref, r, v, a_c = exp(cs_last).
//   2. G = C B^T (tcgen05) -> masked bf16 tril(G) in shared memory.
//   3. Eight 16-token steps through a 3-buffer ring (full/empty mbarriers):
//      all threads build wx (hi, lo) for step k while thread 0 issues step
//      k-1's S_c += wx^T B and Y += tril(G)[:, step] wx on the tensor cores.
//   4. Look-back: if the predecessor chunk's inclusive state is published,
//      read it; else publish (S_c, a_c) as this chunk's aggregate first, then
//      walk back (32 predecessors per poll) to the nearest published inclusive
//      state (or the init state) and apply h <- a_k h + S_k forward, the
//      recurrence's own order, so the result is independent of the walk.
//      Publish h_{c+1} = a_c h_c + S_c; the last chunk writes final_state.
//      Publication: each thread writes its part, then adds 1 to the unit's
//      counter with release semantics (no fence, no barrier); a reader that
//      acquires the full count sees every part.
//   5. Y += C (e^ref h_c)^T (h as hi + lo), then y = r_i Y + D x, staged in
//      shared memory and written by TMA.
//
// A chunk whose span exceeds 120 (an extreme decay inside one chunk: the
// factors would leave range) keeps steps 1-4 with the decay referenced to the
// chunk end (v_j = exp(cs_last - cs_j) <= 1) and replaces the rank-one diagonal
// block by the quadratic form itself: per head, the masked decayed matrix
//   M_ij = G_ij exp(cs_i - cs_j) dt_j  (j <= i),
// every factor at most 1 apart from G, formed from G in TMEM and multiplied
// with x as loaded (exact in bf16) on the tensor cores, and the off-diagonal
// part C h_c^T in a second accumulator scaled by exp(cs_i) <= 1:
//   y_i = (M x)_i + exp(cs_i) C_i . h_c + D x_i.
//
// Forward progress: CTAs take their unit from an atomic ticket in chunk-major
// order (after allocating tensor memory), so every unit a CTA waits on belongs
// to a CTA that started earlier, and no CTA waits before it has published its
// aggregate or its inclusive state.  Every wait is bounded (%globaltimer); a
// wait that gives up sets the device error word and the CTA leaves, which
// makes its successors give up too instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "ssd_internal.cuh"
#include "ssd_ptx.cuh"

namespace ssd {

namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr int kRows = 128;                 // tokens per tile, TMEM lanes
constexpr int kSlab = 64 * 2 * kRows;      // 64 bf16 columns x 128 rows = 16 KiB
constexpr float kSpanMax = 120.f;          // widest in-chunk cs range of the factored path

enum : uint32_t { kFlagNone = 0, kFlagAggregate = 1, kFlagInclusive = 2 };
enum { kCtrTicket = 0, kCtrCount = 4 };

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Publication flag: a release store by one thread after a barrier, which
// orders every participating thread's earlier writes before the flag.
__device__ __forceinline__ void st_release_flag(uint32_t *p)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(1u) : "memory");
}

// Fire-and-forget increment that orders this thread's earlier writes before it.
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

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

// hi = bf16(f), lo = bf16(f - hi), 8 values
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

// A unit's aggregate (inclusive) state is published once its aggcnt (inclcnt)
// reaches the CTA's thread count: every thread adds 1 with release semantics
// after writing its own part, so an acquiring reader that sees the full count
// sees every part.
struct FusedArgs {
    float *agg;          // [units][128][NS] aggregate chunk states S_c
    float *incl;         // [units][128][NS] inclusive states h_{c+1}
    float *alpha;        // [units][2] chunk decays a_c per head of the block
    uint32_t *aggcnt;    // [units] aggregate publication count
    uint32_t *inclcnt;   // [units] inclusive publication count (counters follow)
    uint32_t *counters;  // ticket
};

// Named barrier `id` over `n` threads (id 0 with the whole CTA is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// One CTA per SM: its shared memory (137 KiB at dstate 64, 217 KiB at 128) leaves
// no room for a second, so the registers are not capped for one.  Persistent: the
// CTA takes tickets one after another until `units` are handed out, its TMEM
// allocated once, its barriers initialised afresh for every unit.
template <int NS, bool kPacked>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_fused_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bmap,
                 const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap ymap, Problem pr,
                 FusedArgs fa, int units)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_ld, bar_c, bar_g, bar_w, bar_full[3], bar_empty[3];
    __shared__ uint32_t tmem_slot, s_ticket;
    __shared__ float warp_tot[8], warp_mn[8], warp_mx[8];
    __shared__ float cs[2 * kRows], dtv[2 * kRows];
    __shared__ float vw[2 * kRows];    // v_j dt_j (0 past the chunk end)
    __shared__ float rs[2 * kRows];    // r_i
    __shared__ float s_alpha[2], s_sfac[2], s_yscale[2];
    __shared__ int s_fail, s_mode, s_stop;

    constexpr int NSL = NS / 64;        // 64-wide slabs of the state dimension
    const uint64_t lim = pr.wait_ns;    // limit of every bounded wait
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;       // TMEM lane quarter this warp may access
    const int half = warp >> 2;         // which head / half of the columns this warp handles
    const int P = pr.headdim, HB = 128 / P, H = pr.nheads, L = pr.seqlen;
    const int nhb = H / HB, nc = pr.nchunks;

    // TMEM first, tickets second: a CTA never holds a ticket (that others may wait
    // on) while it is itself still waiting for resources.  A CTA takes its next
    // ticket only after finishing its unit, so every smaller ticket is finished or
    // held by a running unit: the look-back always ends.
    if (warp == 0) tmem_alloc(&tmem_slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t col_y = 0, col_st = 128;   // Y (G first), chunk state
    for (;;) {
    if (tid == 0) {
        s_ticket = atomicAdd(fa.counters + kCtrTicket, 1u);
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_c, 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_w, 1);
        for (int k = 0; k < 3; ++k) {
            mbar_init(&bar_full[k], kThreads / 32);  // one arrival per warp
            mbar_init(&bar_empty[k], 1);
        }
        mbar_fence_init();
        s_fail = 0;
    }
    __syncthreads();
    if (s_ticket >= (uint32_t)units) break;  // the same value for every thread

    // chunk-major unit order: every predecessor chunk has a smaller ticket.  (tt, tb):
    // TMA coordinates of the first token, whose global index is tb * seqlen + tt
    // (packed sequences sit in one batch row); units of one (b, hb) are consecutive
    // in chunk order
    const int ticket = (int)s_ticket;
    int c, b, hb, tt, tb, len, lastflag = 0;
    size_t unit;
    if constexpr (kPacked) {
        const int k = ticket / nhb;
        hb = ticket - k * nhb;
        const int4 d0 = __ldg(reinterpret_cast<const int4 *>(pr.chunks + k));
        const int4 d1 = __ldg(reinterpret_cast<const int4 *>(pr.chunks + k) + 1);
        b = d0.x;
        c = d0.y;
        tt = d0.w;
        tb = 0;
        len = d1.x;
        lastflag = d1.y;
        unit = (size_t)hb * pr.total_chunks + d0.z;
    } else {
        c = ticket / (pr.batch * nhb);
        const int rest = ticket - c * (pr.batch * nhb);
        b = rest / nhb;
        hb = rest - b * nhb;
        tt = c * pr.chunk;
        tb = b;
        len = min(pr.chunk, L - tt);
        unit = ((size_t)b * nhb + hb) * nc + c;
    }
    const int h0 = hb * HB, g = h0 / (H / pr.ngroups);

    uint8_t *base = align1024(smem_raw);
    uint8_t *xs = base;                              // x: 2 MN blocks x 16 KiB
    uint8_t *bs = xs + 2 * kSlab;                    // B, later C again: NSL slabs
    uint8_t *cm = bs + NSL * kSlab;                  // C, then tril(G) (2 slabs), later y staging
    uint8_t *rr = cm + 2 * kSlab;                    // wx ring: 3 x (hi 4 KiB | lo 4 KiB)
    uint8_t *hh_s = NS == 64 ? cm : rr + 3 * 8192;   // h hi | lo (NSL slabs each)
    uint8_t *gl = hh_s + 2 * NSL * kSlab;            // tril(G) lo (2 slabs)

    if (tid == 0) {
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&bmap);
        tma_prefetch_desc(&cmap);
        mbar_expect_tx(&bar_ld, (uint32_t)((2 + 2 * NSL) * kSlab));
        for (int k = 0; k < 2; ++k) tma_load_3d(xs + k * kSlab, &xmap, &bar_ld, hb * 128 + 64 * k, tt, tb);
        for (int s = 0; s < NSL; ++s) {
            tma_load_3d(bs + s * kSlab, &bmap, &bar_ld, g * NS + 64 * s, tt, tb);
            tma_load_3d(cm + s * kSlab, &cmap, &bar_ld, g * NS + 64 * s, tt, tb);
        }
        // the predecessor's inclusive state (or the init state) into L2 ahead of the look-back:
        // with many units per chain position, the predecessor finished long ago and its
        // state (written back from L2 since) would otherwise come from DRAM
        if (c > 0)
            bulk_prefetch_l2(fa.incl + (unit - 1) * (size_t)kRows * NS, (uint32_t)(kRows * NS * sizeof(float)));
        else if (pr.init_state)
            bulk_prefetch_l2(pr.init_state + ((size_t)b * H + h0) * P * NS, (uint32_t)(kRows * NS * sizeof(float)));
    }

    // ---- segment sums, span, reference, factors: warps 0-3 head 0, warps 4-7 head 1
    bool fast;
    {
        const int hh = half, t = tid & 127;
        const bool active = hh < HB;
        const float a = active ? __ldg(pr.A + h0 + hh) : 0.f;
        const float d = (active && t < len) ? __ldg(pr.dt + ((size_t)tb * L + tt + t) * H + h0 + hh) : 0.f;
        const float din =  // input scale
            pr.dtin ? ((active && t < len) ? __ldg(pr.dtin + ((size_t)tb * L + tt + t) * H + h0 + hh) : 0.f) : d;
        float v = d * a;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) warp_tot[warp] = v;
        __syncthreads();
        for (int w = half * 4; w < warp; ++w) v += warp_tot[w];
        // range of cs over the chunk's tokens
        float mn = t < len ? v : 3.0e38f, mx = t < len ? v : -3.0e38f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (lane == 0) {
            warp_mn[warp] = mn;
            warp_mx[warp] = mx;
        }
        cs[hh * kRows + t] = v;
        dtv[hh * kRows + t] = din;
        __syncthreads();
        float lo_[2], hi_[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            lo_[k] = fminf(fminf(warp_mn[4 * k], warp_mn[4 * k + 1]), fminf(warp_mn[4 * k + 2], warp_mn[4 * k + 3]));
            hi_[k] = fmaxf(fmaxf(warp_mx[4 * k], warp_mx[4 * k + 1]), fmaxf(warp_mx[4 * k + 2], warp_mx[4 * k + 3]));
        }
        fast = (hi_[0] - lo_[0] <= kSpanMax) && (HB == 1 || hi_[1] - lo_[1] <= kSpanMax);
        const float cl = cs[hh * kRows + len - 1];
        const float ref = 0.5f * ((hh == 0 ? lo_[0] : lo_[1]) + (hh == 0 ? hi_[0] : hi_[1]));
        const float refw = fast ? ref : cl, refy = fast ? ref : 0.f;
        if (active) {
            vw[hh * kRows + t] = t < len ? expf(refw - v) * din : 0.f;
            rs[hh * kRows + t] = expf(v - refy);
            if (t == 0) {
                s_alpha[hh] = expf(cl);
                s_sfac[hh] = expf(cl - refw);
                s_yscale[hh] = expf(refy);
            }
        }
    }

    bool ok = mbar_wait(&bar_ld, 0, lim);
    if (!ok) s_fail = 1;
    __syncthreads();
    ok = !s_fail;

    // ---- G = C B^T, then the masked bf16 tril(G) over C
    if (ok && tid == 0) {
        tc_fence_after();
        constexpr uint32_t id_g = idesc_bf16(128, 128, 0, 0);
        for (int ks = 0; ks < NS / 16; ++ks) {
            const uint32_t off = (ks / 4) * kSlab + (ks % 4) * 32;
            mma_bf16(tmem + col_y, sdesc_sw128(smem_u32(cm) + off, 16, 1024), sdesc_sw128(smem_u32(bs) + off, 16, 1024),
                     id_g, ks > 0);
        }
        mma_commit(&bar_g);
    }
    if (ok && !mbar_wait(&bar_g, 0, lim)) s_fail = 1;
    __syncthreads();
    ok = !s_fail;
    tc_fence_after();
    const int m = quarter * 32 + lane;   // TMEM row of this thread: token i, or (head, headdim)
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    if (ok && fast) {
        // tril(G) as two bf16 terms (hi = bf16(G), lo = bf16(G - hi)): at dstate 128 a
        // single rounding of G alone costs up to ~2% of RMS(y) where dt is large
        for (int jb = 2 * half; jb < 2 * half + 2; ++jb) {
            uint8_t *dst = cm + (jb >> 1) * kSlab, *dstl = gl + (jb >> 1) * kSlab;
            const int q0 = (jb & 1) * 4;
            if (jb > quarter) {  // every row of this warp is above the diagonal
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    *reinterpret_cast<uint4 *>(dst + sw128(m, q0 + u)) = z;
                    *reinterpret_cast<uint4 *>(dstl + sw128(m, q0 + u)) = z;
                }
                continue;
            }
            float gv[32];
            tmem_ld32(tmem + lane_base + col_y + jb * 32, gv);
            if (jb == quarter) {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (jb * 32 + k > m) gv[k] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint4 hi, lo;
                split8(gv + 8 * u, hi, lo);
                *reinterpret_cast<uint4 *>(dst + sw128(m, q0 + u)) = hi;
                *reinterpret_cast<uint4 *>(dstl + sw128(m, q0 + u)) = lo;
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    if constexpr (NS == 128) {
        // ---- wx = v dt x for all 128 tokens at once: hi in place over x, lo over the
        // h operand region (unused until the look-back); then every chunk-state and
        // diagonal-block MMA in one batch.  x itself comes back by TMA for the D x term.
        uint8_t *wlo = hh_s;
        if (ok) {
#pragma unroll 2
            for (int r = 0; r < (2 * kRows * 8) / kThreads; ++r) {
                const int idx = tid + kThreads * r;  // 16-byte chunk: (64-column block, token, 8 columns)
                const int mb = idx >> 10, j = (idx >> 3) & 127, qq = idx & 7;
                const float w = vw[(P == 64 ? mb : 0) * kRows + j];
                uint4 *ptr = reinterpret_cast<uint4 *>(xs + mb * kSlab + sw128(j, qq));
                const uint4 xv = *ptr;
                const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
                float f[8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 t = __bfloat1622float2(x2[u]);
                    f[2 * u] = t.x * w;
                    f[2 * u + 1] = t.y * w;
                }
                uint4 hi, lo;
                split8(f, hi, lo);
                *ptr = hi;
                *reinterpret_cast<uint4 *>(wlo + mb * kSlab + sw128(j, qq)) = lo;
            }
        }
        fence_async_smem();
        __syncthreads();
        if (ok && tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_s = idesc_bf16(128, NS, 1, 1);
            constexpr uint32_t id_d = idesc_bf16(128, 128, 0, 1);
            for (int k = 0; k < kRows / 16; ++k) {
                const uint64_t whi = sdesc_sw128(smem_u32(xs) + k * 2048, kSlab, 1024);
                const uint64_t wlw = sdesc_sw128(smem_u32(wlo) + k * 2048, kSlab, 1024);
                const uint64_t bd = sdesc_sw128(smem_u32(bs) + k * 2048, kSlab, 1024);
                mma_bf16(tmem + col_st, whi, bd, id_s, k > 0);
                mma_bf16(tmem + col_st, wlw, bd, id_s, 1);
                if (fast) {
                    const uint32_t goff = (k >> 2) * kSlab + (k & 3) * 32;
                    const uint64_t ad = sdesc_sw128(smem_u32(cm) + goff, 16, 1024);
                    const uint64_t adl = sdesc_sw128(smem_u32(gl) + goff, 16, 1024);
                    mma_bf16(tmem + col_y, ad, whi, id_d, k > 0);
                    mma_bf16(tmem + col_y, ad, wlw, id_d, 1);
                    mma_bf16(tmem + col_y, adl, whi, id_d, 1);
                }
            }
            mma_commit(&bar_empty[0]);
        }
        if (ok && !mbar_wait(&bar_empty[0], 0, lim)) s_fail = 1;
    } else {
    // ---- eight 16-token steps through a 3-buffer ring: every thread builds its
    // 16-byte chunk of wx (hi, lo) for step k, each warp then arrives once on
    // full[k % 3]; after its own chunk thread 0 issues step k-1 (S_c += wx^T B ;
    // Y += tril(G)[:, step] wx) and commits it to empty[(k-1) % 3], which the
    // buffer's next writers wait on.
    if (ok) {
        const int mb = tid >> 7, row = (tid >> 3) & 15, qq = tid & 7;
        const float *vh = vw + (P == 64 ? mb : 0) * kRows;
        auto issue = [&](int k) {
            const int bb = k % 3;
            if (!mbar_wait(&bar_full[bb], (k / 3) & 1, lim)) return false;
            tc_fence_after();
            const uint32_t buf = smem_u32(rr) + bb * 8192;
            constexpr uint32_t id_s = idesc_bf16(128, NS, 1, 1);
            const uint64_t bd = sdesc_sw128(smem_u32(bs) + k * 2048, kSlab, 1024);
            mma_bf16(tmem + col_st, sdesc_sw128(buf, 2048, 1024), bd, id_s, k > 0);
            mma_bf16(tmem + col_st, sdesc_sw128(buf + 4096, 2048, 1024), bd, id_s, 1);
            if (fast) {
                constexpr uint32_t id_d = idesc_bf16(128, 128, 0, 1);
                const uint32_t goff = (k >> 2) * kSlab + (k & 3) * 32;
                const uint64_t ad = sdesc_sw128(smem_u32(cm) + goff, 16, 1024);
                const uint64_t adl = sdesc_sw128(smem_u32(gl) + goff, 16, 1024);
                mma_bf16(tmem + col_y, ad, sdesc_sw128(buf, 2048, 1024), id_d, k > 0);
                mma_bf16(tmem + col_y, ad, sdesc_sw128(buf + 4096, 2048, 1024), id_d, 1);
                mma_bf16(tmem + col_y, adl, sdesc_sw128(buf, 2048, 1024), id_d, 1);
            }
            mma_commit(&bar_empty[bb]);
            return true;
        };
        bool good = true;
        for (int k = 0; k < 8 && good; ++k) {
            const int bb = k % 3;
            if (k >= 3 && !mbar_wait(&bar_empty[bb], ((k - 3) / 3) & 1, lim)) good = false;
            if (!good) break;
            uint8_t *buf = rr + bb * 8192;
            const int j = 16 * k + row;
            const float w = vh[j];
            const uint4 xv = *reinterpret_cast<const uint4 *>(xs + mb * kSlab + sw128(j, qq));
            const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
            float f[8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 t = __bfloat1622float2(x2[u]);
                f[2 * u] = t.x * w;
                f[2 * u + 1] = t.y * w;
            }
            uint4 hi, lo;
            split8(f, hi, lo);
            *reinterpret_cast<uint4 *>(buf + mb * 2048 + sw128(row, qq)) = hi;
            *reinterpret_cast<uint4 *>(buf + 4096 + mb * 2048 + sw128(row, qq)) = lo;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_full[bb]);
            // thread 0 issues the previous step once its own chunk of this step is in
            if (tid == 0 && k >= 1) good = issue(k - 1);
        }
        if (good && tid == 0) good = issue(7);
        // the last commit (step 7, buffer 1, its third phase) covers every earlier MMA
        if (good && !mbar_wait(&bar_empty[1], 0, lim)) good = false;
        if (!good) s_fail = 1;
    }
    }
    __syncthreads();
    ok = !s_fail;
    tc_fence_after();
    // x for the D x term: over wx hi for dstate 128, so it comes back (into the dead
    // tril(G) lo region) with C, which the off-diagonal product needs where B was
    uint8_t *xe = NS == 128 ? gl : xs;
    if (ok && tid == 0) {
        mbar_expect_tx(&bar_c, (uint32_t)((NSL + (NS == 128 ? 2 : 0)) * kSlab));
        for (int s = 0; s < NSL; ++s) tma_load_3d(bs + s * kSlab, &cmap, &bar_c, g * NS + 64 * s, tt, tb);
        if (NS == 128)
            for (int k = 0; k < 2; ++k) tma_load_3d(xe + k * kSlab, &xmap, &bar_c, hb * 128 + 64 * k, tt, tb);
    }

    // ---- state passing by decoupled look-back; this thread: row m = (head, headdim),
    // state columns [n0, n0 + NS/2)
    const int hh_m = m / P, p_m = m % P;
    const size_t ustride = (size_t)kRows * NS;
    const int n0 = half * (NS / 2);
    // published states: [NS/4][128 rows][4] per unit (a warp moves 512 contiguous
    // bytes); the float4 holding columns [n, n + 4) of row m sits at (n / 4) * kRows + m
    const size_t row_off = (size_t)(n0 / 4) * kRows * 4 + (size_t)m * 4;
    const float sfac = s_sfac[hh_m];
    if (ok && tid == 0) {
        int mode = 0;  // 0: chunk 0, 1: predecessor inclusive ready, 2: look back
        if (c > 0) mode = ld_acquire(fa.inclcnt + unit - 1) == kThreads ? 1 : 2;
        s_mode = mode;
    }
    __syncthreads();
    const int mode = s_mode;
    if (ok && mode == 2) {
        // publish the aggregate (S_c, a_c) before waiting on anyone
        float4 *dst = reinterpret_cast<float4 *>(fa.agg + unit * ustride + row_off);
        for (int cc = 0; cc < NS / 2; cc += 32) {
            float v[32];
            tmem_ld32(tmem + lane_base + col_st + n0 + cc, v);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                __stcg(dst + (cc / 4 + u) * kRows, make_float4(sfac * v[4 * u], sfac * v[4 * u + 1],
                                                                             sfac * v[4 * u + 2], sfac * v[4 * u + 3]));
        }
        if (tid < HB) fa.alpha[unit * 2 + tid] = s_alpha[tid];
        if ((long long)unit != pr.withhold) red_release_add(fa.aggcnt + unit, 1u);
        if (warp == 0) {
            // Walk back, 32 predecessors per poll: stop at the nearest chunk whose
            // inclusive state is published (or before chunk 0: the init state);
            // every chunk in between must have published its aggregate.
            int top = c - 1, stop = -1;
            const uint64_t tstart = globaltimer();
            bool timed_out = false;
            for (;;) {
                const int k = top - lane;
                uint32_t f = kFlagInclusive;  // before chunk 0: the init state
                if (k >= 0) {
                    const size_t uk = unit - (c - k);
                    f = ld_acquire(fa.inclcnt + uk) == kThreads ? kFlagInclusive
                        : (ld_acquire(fa.aggcnt + uk) == kThreads ? kFlagAggregate : kFlagNone);
                }
                const uint32_t end_mask = __ballot_sync(0xffffffffu, f == kFlagInclusive);
                const uint32_t none_mask = __ballot_sync(0xffffffffu, f == kFlagNone);
                const uint32_t before = end_mask ? (end_mask & (0u - end_mask)) - 1u : 0xffffffffu;
                if ((none_mask & (end_mask ? before : 0xffffffffu)) == 0u) {
                    if (end_mask) {
                        stop = top - (__ffs(end_mask) - 1);  // -1: the init state
                        break;
                    }
                    top -= 32;  // 32 aggregates, keep walking
                    continue;
                }
                // every lane must take the same exit: the next pass's ballots need all 32
                if (__any_sync(0xffffffffu, globaltimer() - tstart > lim)) {
                    timed_out = true;
                    break;
                }
                __nanosleep(64);
            }
            if (lane == 0) {
                s_stop = stop;
                if (timed_out) s_fail = 1;
            }
        }
        __syncthreads();
        ok = !s_fail;
    }

    if (ok) {
        // h_c in the recurrence's own order: start from the stop chunk's inclusive
        // state (or the init state) and apply h <- a_k h + S_k for each later chunk,
        // so the result does not depend on how far the walk went
        const int stop = mode == 2 ? s_stop : c - 1;   // mode 0: c - 1 = -1, the init state
        const float a_own = s_alpha[hh_m], ysc = s_yscale[hh_m];
        const int hg = h0 + hh_m;
        const float *init = pr.init_state ? pr.init_state + (((size_t)b * H + hg) * P + p_m) * NS + n0 : nullptr;
        // the entry state (the stop chunk's inclusive state, or the init state) for all of
        // this thread's columns, every load issued before any is used: one round trip
        float4 ent[NS / 8];
        {
            const float4 *src = stop >= 0 ? reinterpret_cast<const float4 *>(fa.incl + (unit - (c - stop)) * ustride + row_off)
                                          : reinterpret_cast<const float4 *>(init);
            const int qs = stop >= 0 ? kRows : 1;
#pragma unroll
            for (int q = 0; q < NS / 8; ++q) ent[q] = src ? __ldcg(src + q * qs) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int cc = 0; cc < NS / 2; cc += 32) {
            float acc[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = ent[cc / 4 + q];
                acc[4 * q] = v.x;
                acc[4 * q + 1] = v.y;
                acc[4 * q + 2] = v.z;
                acc[4 * q + 3] = v.w;
            }
            int k = stop + 1;
            for (; k + 1 < c; k += 2) {  // two aggregates per round trip
                const size_t u = unit - (c - k);
                const float a0 = __ldcg(fa.alpha + u * 2 + hh_m), a1 = __ldcg(fa.alpha + (u + 1) * 2 + hh_m);
                const float4 *s0 = reinterpret_cast<const float4 *>(fa.agg + u * ustride + row_off + cc * kRows);
                const float4 *s1 = reinterpret_cast<const float4 *>(fa.agg + (u + 1) * ustride + row_off + cc * kRows);
                float4 v0[8], v1[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    v0[q] = __ldcg(s0 + q * kRows);
                    v1[q] = __ldcg(s1 + q * kRows);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    acc[4 * q] = fmaf(a1, fmaf(a0, acc[4 * q], v0[q].x), v1[q].x);
                    acc[4 * q + 1] = fmaf(a1, fmaf(a0, acc[4 * q + 1], v0[q].y), v1[q].y);
                    acc[4 * q + 2] = fmaf(a1, fmaf(a0, acc[4 * q + 2], v0[q].z), v1[q].z);
                    acc[4 * q + 3] = fmaf(a1, fmaf(a0, acc[4 * q + 3], v0[q].w), v1[q].w);
                }
            }
            if (k < c) {
                const size_t u = unit - (c - k);
                const float a = __ldcg(fa.alpha + u * 2 + hh_m);
                const float4 *src = reinterpret_cast<const float4 *>(fa.agg + u * ustride + row_off + cc * kRows);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 v = __ldcg(src + q * kRows);
                    acc[4 * q] = fmaf(a, acc[4 * q], v.x);
                    acc[4 * q + 1] = fmaf(a, acc[4 * q + 1], v.y);
                    acc[4 * q + 2] = fmaf(a, acc[4 * q + 2], v.z);
                    acc[4 * q + 3] = fmaf(a, acc[4 * q + 3], v.w);
                }
            }
            {  // e^ref h_c -> bf16 hi / lo operand slabs (row m); ref = 0 in a wide unit
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float f[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) f[u] = ysc * acc[8 * q + u];
                    uint4 hi, lo;
                    split8(f, hi, lo);
                    const int n = n0 + cc + 8 * q;
                    const uint32_t o = (n / 64) * kSlab + sw128(m, (n % 64) / 8);
                    *reinterpret_cast<uint4 *>(hh_s + o) = hi;
                    *reinterpret_cast<uint4 *>(hh_s + NSL * kSlab + o) = lo;
                }
            }
            // h_{c+1} = a_c h_c + S_c
            float sc[32];
            tmem_ld32(tmem + lane_base + col_st + n0 + cc, sc);
#pragma unroll
            for (int k = 0; k < 32; ++k) sc[k] = fmaf(a_own, acc[k], sfac * sc[k]);
            float4 *dst = reinterpret_cast<float4 *>(fa.incl + unit * ustride + row_off + cc * kRows);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                __stcg(dst + q * kRows, make_float4(sc[4 * q], sc[4 * q + 1], sc[4 * q + 2], sc[4 * q + 3]));
            if ((kPacked ? lastflag != 0 : c == nc - 1) && pr.final_state) {
                float4 *fo = reinterpret_cast<float4 *>(pr.final_state + (((size_t)b * H + hg) * P + p_m) * NS + n0 + cc);
#pragma unroll
                for (int q = 0; q < 8; ++q) fo[q] = make_float4(sc[4 * q], sc[4 * q + 1], sc[4 * q + 2], sc[4 * q + 3]);
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if constexpr (NS == 128) {
        if (!fast) {
            // A wide unit has no rank-one decay.  Its diagonal block takes, per head, the
            // masked decayed matrix M[i][j] = G_ij e^(cs_i - cs_j) dt_j (j <= i; every factor
            // <= 1 apart from G) as bf16 hi (over the dead wx hi) and lo (over C, whose G is
            // done) K-major operands, formed from G in TMEM, and Y_diag[:, hh P ..] = M_hh x_hh
            // accumulates in S_c's columns (consumed above), so G stays whole for the next
            // head; x is exact in bf16.  This thread: row m, columns [64 half, 64 half + 64).
            for (int hh = 0; hh < HB; ++hh) {
                if (ok) {
                    const float csm = cs[hh * kRows + m];
#pragma unroll 1
                    for (int jb = 0; jb < 4; ++jb) {
                        const int j0 = 64 * half + 16 * jb;
                        uint8_t *dh = xs + half * kSlab, *dl = cm + half * kSlab;
                        uint4 hi[2], lo[2];
                        if (j0 <= 32 * quarter + 31) {  // warp-uniform: some row of this warp reaches j0
                            float gv[16];
                            tmem_ld16(tmem + lane_base + col_y + j0, gv);
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                const int j = j0 + k;
                                const float w = __expf(csm - cs[hh * kRows + j]) * dtv[hh * kRows + j];
                                gv[k] = j <= m ? gv[k] * w : 0.f;
                            }
                            split8(gv, hi[0], lo[0]);
                            split8(gv + 8, hi[1], lo[1]);
                        } else {
                            hi[0] = hi[1] = lo[0] = lo[1] = make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            *reinterpret_cast<uint4 *>(dh + sw128(m, 2 * jb + u)) = hi[u];
                            *reinterpret_cast<uint4 *>(dl + sw128(m, 2 * jb + u)) = lo[u];
                        }
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncthreads();
                if (ok && tid == 0) {
                    if (hh == 0 && !mbar_wait(&bar_c, 0, lim)) {
                        s_fail = 1;
                    } else {
                        tc_fence_after();
                        const uint32_t id_w = idesc_bf16(128, P, 0, 1);
                        for (int k = 0; k < kRows / 16; ++k) {
                            const uint32_t goff = (k >> 2) * kSlab + (k & 3) * 32;
                            const uint64_t xd = sdesc_sw128(smem_u32(xe) + hh * kSlab + k * 2048, kSlab, 1024);
                            mma_bf16(tmem + col_st + hh * P, sdesc_sw128(smem_u32(xs) + goff, 16, 1024), xd, id_w, k > 0);
                            mma_bf16(tmem + col_st + hh * P, sdesc_sw128(smem_u32(cm) + goff, 16, 1024), xd, id_w, 1);
                        }
                        mma_commit(&bar_w);
                    }
                }
                __syncthreads();
                ok = ok && !s_fail;
                // the next head's M goes where this one was: wait for its MMAs
                if (ok && !mbar_wait(&bar_w, hh & 1, lim)) s_fail = 1;
                __syncthreads();
                ok = ok && !s_fail;
                tc_fence_after();
            }
        }
    }
    if (ok && tid == 0) {
        // Y += C (e^ref h_c)^T; a wide unit's off-diagonal part starts its own accumulator over G
        if (!mbar_wait(&bar_c, 0, lim)) {
            s_fail = 1;
        } else {
            tc_fence_after();
            constexpr uint32_t id_o = idesc_bf16(128, 128, 0, 0);
            for (int ks = 0; ks < NS / 16; ++ks) {
                const uint32_t off = (ks / 4) * kSlab + (ks % 4) * 32;
                const uint64_t ad = sdesc_sw128(smem_u32(bs) + off, 16, 1024);
                mma_bf16(tmem + col_y, ad, sdesc_sw128(smem_u32(hh_s) + off, 16, 1024), id_o, fast || ks > 0);
                mma_bf16(tmem + col_y, ad, sdesc_sw128(smem_u32(hh_s) + NSL * kSlab + off, 16, 1024), id_o, 1);
            }
            mma_commit(&bar_g);
        }
    }
    // publish h_{c+1} (written above) now that the off-diagonal MMA is running:
    // the release waits for this thread's stores, off the critical path
    if (ok && (long long)unit != pr.withhold) red_release_add(fa.inclcnt + unit, 1u);
    __syncthreads();
    ok = ok && !s_fail;
    if (ok && !mbar_wait(&bar_g, 1, lim)) s_fail = 1;
    __syncthreads();
    ok = ok && !s_fail;
    tc_fence_after();

    // ---- y = r_i Y + D x; this thread: row i, 64 of the 128 (head, headdim) columns
    // full 128-row tiles: staged in shared memory, TMA store (a packed sequence's partial
    // chunk is stored row by row: the rows after it belong to the next sequence)
    const bool tma_out = pr.chunk == kRows && (!kPacked || len == kRows);
    uint8_t *ystage = cm;
    if (ok) {
        const int i = m, col0 = half * 64;
        const int hh = col0 / P, h = h0 + hh;
        const float r = rs[hh * kRows + i];
        const float Dh = pr.D ? __ldg(pr.D + h) : 0.f;
        for (int pc = 0; pc < 64; pc += 32) {
            const int col = col0 + pc;
            float yv[32];
            tmem_ld32(tmem + lane_base + col_y + col, yv);
            if (!fast) {  // a wide unit: y = Y_diag + r Y_off + D x, r = e^cs
                float yd[32];
                tmem_ld32(tmem + lane_base + col_st + col, yd);
#pragma unroll
                for (int k = 0; k < 32; ++k) yv[k] = fmaf(r, yv[k], yd[k]);
            }
            const float rr = fast ? r : 1.f;
            uint4 outv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xe + half * kSlab + sw128(i, pc / 8 + u));
                const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
                float o[8];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float2 xf = __bfloat1622float2(x2[v]);
                    o[2 * v] = fmaf(Dh, xf.x, rr * yv[8 * u + 2 * v]);
                    o[2 * v + 1] = fmaf(Dh, xf.y, rr * yv[8 * u + 2 * v + 1]);
                }
                outv[u] = pack8(o);
            }
            if (tma_out) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4 *>(ystage + half * kSlab + sw128(i, pc / 8 + u)) = outv[u];
            } else if (i < len) {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(pr.y) +
                                                       (((size_t)tb * L + tt + i) * H + h0) * P + col);
#pragma unroll
                for (int u = 0; u < 4; ++u) dst[u] = outv[u];
            }
        }
    }
    if (tma_out) {
        fence_async_smem();
        __syncthreads();
        if (ok && tid == 0) {
            for (int k = 0; k < 2; ++k) tma_store_3d(&ymap, ystage + k * kSlab, hb * 128 + 64 * k, tt, tb);
            bulk_commit();
            bulk_wait_read_all();
        }
    }
    if (!ok && tid == 0) atomicOr(pr.err_word, kDevErrTimeout);
    // the unit is done: its shared memory, barriers and TMEM columns are free again;
    // a wait that gave up ends this CTA's work
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();
    }
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// dstate 64, persistent.  One CTA per SM takes units (chunk-major tickets, as
// above) one after another and keeps two of them in flight: two shared-memory
// stages of 96 KiB and two TMEM slots, unit it using stage and slot it & 1.
// Warp roles:
//   warp 0      tickets; TMA loads of dt, x, B and C into a free stage;
//   warp 1      G = C B^T; the chunk-state MMAs slice by slice, committed on
//               their own (the chain waits for S_c only); then the diagonal
//               block Y = tril(G) wx once tril(G) is in (hi and lo: 3 MMAs);
//   warps 2-5   segment sums and factors, wx (hi, lo) in 16-token slices, then
//               tril(G) as hi and lo bf16 into TMEM (after wx, so S_c does not
//               wait for it);
//   warps 6-9   team 0 (the units of stage 0), warps 10-13 team 1 (stage 1):
//               look-back for h_c (publishing S_c as the aggregate if the walk
//               is still waiting when S_c is ready), h_{c+1} published, then
//               (once the diagonal block is done with wx) x brought into the
//               staging region by TMA, the h operand and the off-diagonal MMA
//               Y += C (e^ref h_c)^T, y = r Y + D x, and the TMA store of y; a
//               wide unit's outputs instead (see the team's code).
// Each role walks its units in ticket order, so the forward-progress argument
// of the one-unit kernel holds: the smallest unfinished ticket only waits on
// finished units.  Stage s, 96 KiB: [0, 32K) x -> wx hi -> h hi | lo;
// [32K, 64K) wx lo -> x -> y (staging); [64K, 80K) B; [80K, 96K) C; after the
// two stages, 2 KiB of dt per stage.  TMEM: slot s at column 256 s holds Y
// [0,128) and S_c [128,192); tril(G) hi [192,256) and lo [448,512) serve the
// unit the front and the MMA warp are on (a unit's G commit follows the
// previous unit's diagonal MMAs from the same thread, so the front may then
// overwrite them).  The stage's x, B and C are reloaded as soon as the
// off-diagonal MMA completes; the wx-lo region waits for the y store.
// Per-unit scalars and the info and seg barriers have four sets (it & 3): a
// team may still read them after its stage has been handed to the next unit.
// ---------------------------------------------------------------------------
constexpr int kPipeThreads = 16 * 32;
constexpr int kStageBytes = 6 * kSlab;
constexpr int kDtBytes = kRows * 4 * sizeof(float);  // dt box: 128 tokens x 4 heads
constexpr int kSlices = kRows / 16;  // wx is built, and consumed by the MMAs, 16 tokens at a time
enum { kWarpLoad = 0, kWarpMma = 1, kWarpFront = 2, kWarpState = 6, kWarpPub = 14 };
enum { kBarFront = 1, kBarTeam0 = 2 };  // team 1 uses barrier 3

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

// A unit: sequence b (a batch element or a packed sequence), chunk c of it, head
// block hb.  (tt, tb) are its TMA coordinates (first token, batch row); the
// global index of its first token is tb * seqlen + tt in both layouts (packed
// sequences sit in one batch row).  Units of one (b, hb) have consecutive
// indices in chunk order, so chunk k of the same sequence is unit - (c - k).
struct PipeUnit {
    int b, hb, c, h0, g, tt, tb, len, last;
    size_t unit;
};

template <bool kPacked>
__device__ __forceinline__ PipeUnit decode_unit(const Problem &pr, int ticket, int nhb)
{
    PipeUnit u;
    if constexpr (kPacked) {  // packed sequences: the chunk table is already chunk-major
        const int k = ticket / nhb;
        u.hb = ticket - k * nhb;
        const int4 d0 = __ldg(reinterpret_cast<const int4 *>(pr.chunks + k));
        const int4 d1 = __ldg(reinterpret_cast<const int4 *>(pr.chunks + k) + 1);
        u.b = d0.x;
        u.c = d0.y;
        u.tt = d0.w;
        u.tb = 0;
        u.len = d1.x;
        u.last = d1.y;
        u.unit = (size_t)u.hb * pr.total_chunks + d0.z;
    } else {
        u.c = ticket / (pr.batch * nhb);
        const int rest = ticket - u.c * (pr.batch * nhb);
        u.b = rest / nhb;
        u.hb = rest - u.b * nhb;
        u.tt = u.c * pr.chunk;
        u.tb = u.b;
        u.len = min(pr.chunk, pr.seqlen - u.tt);
        u.last = 0;  // unit_is_last() derives it from c
        u.unit = ((size_t)u.b * nhb + u.hb) * pr.nchunks + u.c;
    }
    const int HB = 128 / pr.headdim;
    u.h0 = u.hb * HB;
    u.g = u.h0 / (pr.nheads / pr.ngroups);
    return u;
}

template <bool kPacked>
__device__ __forceinline__ bool unit_is_last(const Problem &pr, const PipeUnit &u)
{
    if constexpr (kPacked) return u.last != 0;
    return u.c == pr.nchunks - 1;
}

template <bool kPacked>
__global__ void __launch_bounds__(kPipeThreads, 1)
    ssd_fused_pipe_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bmap,
                      const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap ymap,
                      const __grid_constant__ CUtensorMap dtmap, Problem pr, FusedArgs fa, int units, int dt_tma)
{
    constexpr int NS = 64;
    const uint64_t lim = pr.wait_ns;  // limit of every bounded wait
    extern __shared__ uint8_t smem_raw[];
    // per stage (it & 1): full, free, slot, g, fr, mma, yo; per unit in flight (it & 3): info,
    // seg and the unit's scalars, which the epilogue may still read after the stage is free
    __shared__ __align__(8) uint64_t bar_info[4], bar_seg[4], bar_full[2], bar_dt[2], bar_free[2], bar_slot[2],
        bar_lo[2], bar_g[2], bar_mask[2], bar_slice[2][kSlices], bar_mma[2], bar_yo[2], bar_xe[2], bar_pincl[2],
        bar_pdone[2], bar_wd[2], bar_dg[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int s_tk[4], s_fast[4];
    __shared__ float cs[4][2 * kRows], dtv[4][2 * kRows], vw[4][2 * kRows], rs[4][2 * kRows];
    __shared__ float s_alpha[4][2], s_sfac[4][2], s_ysc[4][2];
    __shared__ float wtot[4][2], wmn[4][2], wmx[4][2];
    __shared__ int s_walk[2][2];
    __shared__ int s_fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;  // TMEM lane of this thread (warps 2-13)
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int P = pr.headdim, HB = 128 / P, H = pr.nheads;
    const int nhb = H / HB;
    // per slot: Y, S_c; tril(G) hi | lo in the columns after each slot's S_c, shared by the units
    const uint32_t col_y = 0, col_st = 128, col_mhi = 192, col_mlo = 448;

    if (warp == kWarpMma) tmem_alloc(&tmem_slot, 512);
    if (tid == 0) {
        for (int k = 0; k < 4; ++k) {
            mbar_init(&bar_info[k], 1);
            mbar_init(&bar_seg[k], 128);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bar_full[k], 1);
            mbar_init(&bar_dt[k], 1);
            mbar_init(&bar_free[k], 1);
            mbar_init(&bar_slot[k], 4);
            mbar_init(&bar_lo[k], 1);
            mbar_init(&bar_g[k], 1);
            mbar_init(&bar_mask[k], 128);
            for (int q = 0; q < kSlices; ++q) mbar_init(&bar_slice[k][q], 128);
            mbar_init(&bar_mma[k], 1);
            mbar_init(&bar_yo[k], 1);
            mbar_init(&bar_xe[k], 1);
            mbar_init(&bar_pincl[k], 4);
            mbar_init(&bar_pdone[k], 1);
            mbar_init(&bar_wd[k], 1);
            mbar_init(&bar_dg[k], 1);
        }
        mbar_fence_init();
        s_fail = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    uint8_t *base = align1024(smem_raw);

    if (warp == kWarpLoad) {
        // ================= tickets and loads
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            tma_prefetch_desc(&bmap);
            tma_prefetch_desc(&cmap);
            tma_prefetch_desc(&ymap);
            int ends = 0;
            if (dt_tma) tma_prefetch_desc(&dtmap);
            for (int it = 0;; ++it) {
                const int s = it & 1, ss = it & 3;
                const uint32_t ph = (it >> 1) & 1;
                bool ok = it < 2 || mbar_wait(&bar_free[s], ph ^ 1, lim);
                const uint32_t t = ok ? atomicAdd(fa.counters + kCtrTicket, 1u) : 0xffffffffu;
                const int tk = t < (uint32_t)units ? (int)t : -1;
                if (!ok) s_fail = 1;
                s_tk[ss] = tk;
                mbar_arrive(&bar_info[ss]);
                if (tk < 0) {
                    // the two teams take alternate units: each needs its own end marker
                    if (++ends == 2 || !ok) break;
                    continue;
                }
                const PipeUnit u = decode_unit<kPacked>(pr, tk, nhb);
                uint8_t *st = base + s * kStageBytes;
                if (dt_tma) {  // dt of the unit's 128 tokens x 4 heads from h0 rounded down to 4
                    mbar_expect_tx(&bar_dt[s], (uint32_t)(kRows * 4 * sizeof(float)));
                    tma_load_3d(base + 2 * kStageBytes + s * kDtBytes, &dtmap, &bar_dt[s], u.h0 & ~3, u.tt, u.tb);
                } else {
                    mbar_arrive(&bar_dt[s]);
                }
                mbar_expect_tx(&bar_full[s], (uint32_t)(4 * kSlab));
                for (int k = 0; k < 2; ++k) tma_load_3d(st + k * kSlab, &xmap, &bar_full[s], u.hb * 128 + 64 * k, u.tt, u.tb);
                tma_load_3d(st + 4 * kSlab, &bmap, &bar_full[s], u.g * NS, u.tt, u.tb);
                tma_load_3d(st + 5 * kSlab, &cmap, &bar_full[s], u.g * NS, u.tt, u.tb);
            }
        }
    } else if (warp == kWarpMma) {
        // ================= G, chunk-state and diagonal-block MMAs
        if (lane == 0) {
            constexpr uint32_t id_g = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_s = idesc_bf16(128, NS, 1, 1);
            constexpr uint32_t id_d = idesc_bf16(128, 128, 0, 1);
            for (int it = 0;; ++it) {
                const int s = it & 1, ss = it & 3;
                const uint32_t ph = (it >> 1) & 1, pq = (it >> 2) & 1;
                if (!mbar_wait(&bar_info[ss], pq, lim)) {
                    s_fail = 1;
                    break;
                }
                if (s_tk[ss] < 0) break;
                const uint32_t slot = tmem + s * 256;
                const uint32_t st = smem_u32(base + s * kStageBytes);
                if (it >= 2 && !mbar_wait(&bar_slot[s], ph ^ 1, lim)) {
                    s_fail = 1;
                    break;
                }
                if (!mbar_wait(&bar_full[s], ph, lim)) {
                    s_fail = 1;
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < NS / 16; ++ks)
                    mma_bf16(slot + col_y, sdesc_sw128(st + 5 * kSlab + ks * 32, 16, 1024),
                             sdesc_sw128(st + 4 * kSlab + ks * 32, 16, 1024), id_g, ks > 0);
                mma_commit(&bar_g[s]);
                // the chunk state slice by slice as the front warps finish wx, committed on its
                // own (the chain waits for it); then the diagonal block once tril(G) is in
                bool okm = true;
                for (int ks = 0; ks < kRows / 16; ++ks) {
                    if (!mbar_wait(&bar_slice[s][ks], ph, lim)) {
                        okm = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = sdesc_sw128(st + 4 * kSlab + ks * 2048, kSlab, 1024);
                    mma_bf16(slot + col_st, sdesc_sw128(st + ks * 2048, kSlab, 1024), bd, id_s, ks > 0);
                    mma_bf16(slot + col_st, sdesc_sw128(st + 2 * kSlab + ks * 2048, kSlab, 1024), bd, id_s, 1);
                }
                if (!okm) {
                    s_fail = 1;
                    break;
                }
                mma_commit(&bar_mma[s]);
                if (!mbar_wait(&bar_mask[s], ph, lim)) {
                    s_fail = 1;
                    break;
                }
                if (s_fast[ss] != 0) {  // written by the front before its bar_mask arrival
                    tc_fence_after();
                    for (int ks = 0; ks < kRows / 16; ++ks) {
                        const uint64_t whi = sdesc_sw128(st + ks * 2048, kSlab, 1024);
                        const uint64_t wlo = sdesc_sw128(st + 2 * kSlab + ks * 2048, kSlab, 1024);
                        mma_bf16_tA(slot + col_y, tmem + col_mhi + ks * 8, whi, id_d, ks > 0);
                        mma_bf16_tA(slot + col_y, tmem + col_mhi + ks * 8, wlo, id_d, 1);
                        mma_bf16_tA(slot + col_y, tmem + col_mlo + ks * 8, whi, id_d, 1);
                    }
                }
                mma_commit(&bar_dg[s]);
            }
        }
    } else if (warp < kWarpState) {
        // ================= segment sums, wx, tril(G)
        const int ft = tid - 32 * kWarpFront, fw = warp - kWarpFront;  // token ft, in warp order
        for (int it = 0;; ++it) {
            const int s = it & 1, ss = it & 3;
            const uint32_t ph = (it >> 1) & 1, pq = (it >> 2) & 1;
            bool ok = mbar_wait(&bar_info[ss], pq, lim);
            const int tk = s_tk[ss];
            if (named_sync_or(kBarFront, 128, !ok)) {
                s_fail = 1;
                break;
            }
            if (tk < 0) break;  // the same ticket for every thread
            const PipeUnit u = decode_unit<kPacked>(pr, tk, nhb);
            uint8_t *st = base + s * kStageBytes;
            const float *dts = reinterpret_cast<const float *>(base + 2 * kStageBytes + s * kDtBytes) + ft * 4 + (u.h0 & 3);
            if (dt_tma) ok = ok && mbar_wait(&bar_dt[s], ph, lim);
            float v[2], d[2], din[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const bool act = hh < HB;
                const float a = act ? __ldg(pr.A + u.h0 + hh) : 0.f;
                d[hh] = (act && ft < u.len)
                            ? (dt_tma ? dts[hh] : __ldg(pr.dt + ((size_t)u.tb * pr.seqlen + u.tt + ft) * H + u.h0 + hh))
                            : 0.f;
                din[hh] = pr.dtin ? ((act && ft < u.len) ? __ldg(pr.dtin + ((size_t)u.tb * pr.seqlen + u.tt + ft) * H + u.h0 + hh) : 0.f)
                                  : d[hh];  // input scale
                v[hh] = d[hh] * a;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t = __shfl_up_sync(0xffffffffu, v[hh], o);
                    if (lane >= o) v[hh] += t;
                }
                if (lane == 31) wtot[fw][hh] = v[hh];
            }
            named_sync(kBarFront, 128);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                for (int w = 0; w < fw; ++w) v[hh] += wtot[w][hh];
                float mn = ft < u.len ? v[hh] : 3.0e38f, mx = ft < u.len ? v[hh] : -3.0e38f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                }
                if (lane == 0) {
                    wmn[fw][hh] = mn;
                    wmx[fw][hh] = mx;
                }
                cs[ss][hh * kRows + ft] = v[hh];
                dtv[ss][hh * kRows + ft] = din[hh];
            }
            named_sync(kBarFront, 128);
            float lo_[2], hi_[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                lo_[hh] = fminf(fminf(wmn[0][hh], wmn[1][hh]), fminf(wmn[2][hh], wmn[3][hh]));
                hi_[hh] = fmaxf(fmaxf(wmx[0][hh], wmx[1][hh]), fmaxf(wmx[2][hh], wmx[3][hh]));
            }
            const bool fast = (hi_[0] - lo_[0] <= kSpanMax) && (HB == 1 || hi_[1] - lo_[1] <= kSpanMax);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (hh >= HB) break;
                const float cl = cs[ss][hh * kRows + u.len - 1];
                const float ref = 0.5f * (lo_[hh] + hi_[hh]);
                const float refw = fast ? ref : cl, refy = fast ? ref : 0.f;
                vw[ss][hh * kRows + ft] = ft < u.len ? expf(refw - v[hh]) * din[hh] : 0.f;
                rs[ss][hh * kRows + ft] = expf(v[hh] - refy);
                if (ft == 0) {
                    s_alpha[ss][hh] = expf(cl);
                    s_sfac[ss][hh] = expf(cl - refw);
                    s_ysc[ss][hh] = expf(refy);
                }
            }
            if (ft == 0) s_fast[ss] = fast ? 1 : 0;
            mbar_arrive(&bar_seg[ss]);
            named_sync(kBarFront, 128);  // every v_j dt_j is in shared memory
            // x in place; the lo region is the staging region of the unit two back: its y is stored
            ok = ok && mbar_wait(&bar_full[s], ph, lim) && (it < 2 || mbar_wait(&bar_lo[s], ph ^ 1, lim));
            // wx = v dt x, hi in place over x, lo at +32K, in 16-token slices: slice
            // ks is rows 16 ks .. 16 ks + 15 of both 64-column slabs (256 chunks)
#pragma unroll 1
            for (int ks = 0; ks < kSlices; ++ks) {
                if (ok) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int idx = ft + 128 * r;
                        const int mb = idx >> 7, j = 16 * ks + ((idx >> 3) & 15), qq = idx & 7;
                        const float w = vw[ss][(P == 64 ? mb : 0) * kRows + j];
                        uint4 *ptr = reinterpret_cast<uint4 *>(st + mb * kSlab + sw128(j, qq));
                        const uint4 xv = *ptr;
                        const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
                        const float2 w2 = make_float2(w, w);
                        float f[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 t = __fmul2_rn(__bfloat1622float2(x2[k]), w2);
                            f[2 * k] = t.x;
                            f[2 * k + 1] = t.y;
                        }
                        uint4 hi, lo;
                        split8(f, hi, lo);
                        *ptr = hi;
                        *reinterpret_cast<uint4 *>(st + 2 * kSlab + mb * kSlab + sw128(j, qq)) = lo;
                    }
                }
                fence_async_smem();
                mbar_arrive(&bar_slice[s][ks]);
            }
            // tril(G) after wx: the chunk state (the chain's next step) does not wait for it
            ok = ok && mbar_wait(&bar_g[s], ph, lim);
            ok = __all_sync(0xffffffffu, ok);  // the TMEM accesses below are warp-collective
            tc_fence_after();
            if (ok && fast) {
                // tril(G) -> hi and lo bf16 pairs (row m, 16 tokens per step) in the shared
                // tril columns.  The previous unit's diagonal MMAs, which read them, are
                // complete: this unit's G commit follows them from the same issuing thread.
                const uint32_t gsrc = tmem + s * 256 + lane_base + col_y;
#pragma unroll 1
                for (int jb = 0; jb < 4; ++jb) {
                    uint32_t ph16[16], pl16[16];
                    if (jb > quarter) {  // every row of this warp is above these columns
#pragma unroll
                        for (int k = 0; k < 16; ++k) ph16[k] = pl16[k] = 0u;
                    } else {
                        float gv[32];
                        tmem_ld32(gsrc + jb * 32, gv);
                        if (jb == quarter) {
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                if (jb * 32 + k > m) gv[k] = 0.f;
                        }
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(gv[2 * k], gv[2 * k + 1]);
                            const float2 hf = __bfloat1622float2(h2);
                            __nv_bfloat162 l2 = __floats2bfloat162_rn(gv[2 * k] - hf.x, gv[2 * k + 1] - hf.y);
                            ph16[k] = *reinterpret_cast<uint32_t *>(&h2);
                            pl16[k] = *reinterpret_cast<uint32_t *>(&l2);
                        }
                    }
                    tmem_st16_async(tmem + lane_base + col_mhi + jb * 16, ph16);
                    tmem_st16_async(tmem + lane_base + col_mlo + jb * 16, pl16);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&bar_mask[s]);
            if (named_sync_or(kBarFront, 128, !ok)) {
                s_fail = 1;
                break;
            }
        }
    } else if (warp >= kWarpPub) {
        // ================= publishers, one per team: release a unit's inclusive state
        // once the team's four warps have stored it, so no team warp stalls on it
        const int team = warp - kWarpPub, s = team;
        if (lane == 0) {
            for (int it = team;; it += 2) {
                const int ss = it & 3;
                const uint32_t ph = (it >> 1) & 1, pq = (it >> 2) & 1;
                if (!mbar_wait(&bar_info[ss], pq, lim)) {
                    s_fail = 1;
                    break;
                }
                const int tk = s_tk[ss];
                if (tk < 0) break;
                if (!mbar_wait(&bar_pincl[s], ph, lim)) {
                    s_fail = 1;
                    break;
                }
                const size_t pu = decode_unit<kPacked>(pr, tk, nhb).unit;
                if (!s_fail && (long long)pu != pr.withhold) red_release_add(fa.inclcnt + pu, 1u);
                mbar_arrive(&bar_pdone[s]);
            }
        }
    } else {
        // ================= two teams, warps 6-9 for the even units (stage 0) and
        // 10-13 for the odd ones (stage 1): look-back for h_c (publishing S_c as the
        // aggregate if the walk is still waiting when S_c is ready), h operand,
        // off-diagonal MMA, inclusive state, then y = r Y + D x staged over the dead
        // wx lo and stored by TMA
        const int team = (warp - kWarpState) >> 2;
        const int tt = tid - 32 * (kWarpState + 4 * team);
        const int bar_team = kBarTeam0 + team;
        const int hh_m = m / P, p_m = m % P;
        const size_t ustride = (size_t)kRows * NS;
        // full 128-row tiles go out by TMA; a packed sequence's partial last chunk is
        // stored row by row, since the rows after it belong to the next sequence
        const bool tma_tiles = pr.chunk == kRows;
        const int s = team;
        uint8_t *st = base + s * kStageBytes;
        const uint32_t slot = tmem + s * 256 + lane_base;
        int nwide = 0;  // commits to bar_wd so far (its phase): the MMA steps of wide units
        for (int it = team;; it += 2) {
            const int ss = it & 3;
            const uint32_t ph = (it >> 1) & 1, pq = (it >> 2) & 1;
            bool ok = mbar_wait(&bar_info[ss], pq, lim);
            const int tk = s_tk[ss];
            if (named_sync_or(bar_team, 128, !ok)) {
                s_fail = 1;
                break;
            }
            if (tk < 0) break;  // the same ticket for every thread
            const PipeUnit u = decode_unit<kPacked>(pr, tk, nhb);
            const int c = u.c;
            const bool tma_out = tma_tiles && (!kPacked || u.len == kRows);
            if (it >= 2 && !mbar_wait(&bar_pdone[s], ph ^ 1, lim)) ok = false;
            // walk back to the nearest inclusive state; -2: S_c became ready first
            // (publish it as the aggregate, then walk on); -3: gave up
            int stop = c - 1;
            if (c > 0) {
                for (int round = 0; round < 2; ++round) {
                    if (tt < 32) {
                        int res = -3, top = c - 1;
                        const uint64_t tstart = globaltimer();
                        for (;;) {
                            const int k = top - lane;
                            uint32_t f = kFlagInclusive;
                            if (k >= 0) {
                                const size_t uk = u.unit - (c - k);
                                f = ld_acquire(fa.inclcnt + uk) != 0u ? kFlagInclusive
                                    : (ld_acquire(fa.aggcnt + uk) != 0u ? kFlagAggregate : kFlagNone);
                            }
                            const uint32_t end_mask = __ballot_sync(0xffffffffu, f == kFlagInclusive);
                            const uint32_t none_mask = __ballot_sync(0xffffffffu, f == kFlagNone);
                            const uint32_t before = end_mask ? (end_mask & (0u - end_mask)) - 1u : 0xffffffffu;
                            if ((none_mask & (end_mask ? before : 0xffffffffu)) == 0u) {
                                if (end_mask) {
                                    res = top - (__ffs(end_mask) - 1);
                                    break;
                                }
                                top -= 32;
                                continue;
                            }
                            // every lane must take the same exit: the next pass's ballots need all 32
                            if (round == 0 && !unit_is_last<kPacked>(pr, u) &&
                                __any_sync(0xffffffffu, mbar_test_wait(&bar_mma[s], ph))) {
                                res = -2;
                                break;
                            }
                            if (__any_sync(0xffffffffu, globaltimer() - tstart > lim)) break;
                            __nanosleep(128);
                        }
                        if (lane == 0) s_walk[team][round] = res;
                    }
                    named_sync(bar_team, 128);
                    const int res = s_walk[team][round];
                    if (res >= -1) {
                        stop = res;
                        break;
                    }
                    if (res == -3) {
                        ok = false;
                        break;
                    }
                    // publish S_c (scaled to the chunk end) as this unit's aggregate
                    ok = mbar_wait(&bar_mma[s], ph, lim) && mbar_wait(&bar_seg[ss], pq, lim);
                    ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
                    tc_fence_after();
                    if (ok) {
                        const float sfac = s_sfac[ss][hh_m];
                        float4 *dst = reinterpret_cast<float4 *>(fa.agg + u.unit * ustride) + m;
                        for (int cc = 0; cc < NS; cc += 32) {
                            float sv[32];
                            tmem_ld32(slot + col_st + cc, sv);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                __stcg(dst + (cc / 4 + q) * kRows,
                                       make_float4(sfac * sv[4 * q], sfac * sv[4 * q + 1], sfac * sv[4 * q + 2],
                                                   sfac * sv[4 * q + 3]));
                        }
                        if (tt < HB) fa.alpha[u.unit * 2 + tt] = s_alpha[ss][tt];
                    }
                    // one release for the whole unit: the barrier orders every
                    // thread's stores before the leader's release store
                    if (!named_sync_or(bar_team, 128, !ok) && tt == 32 && (long long)u.unit != pr.withhold)
                        st_release_flag(fa.aggcnt + u.unit);
                }
            }
            // h_c for row m, in the recurrence's own order
            float acc[NS];
#pragma unroll
            for (int k = 0; k < NS; ++k) acc[k] = 0.f;
            const int hg = u.h0 + hh_m;
            if (ok) {
                const float *init = pr.init_state ? pr.init_state + (((size_t)u.b * H + hg) * P + p_m) * NS : nullptr;
                // published states: [NS/4][128 rows][4] per unit, so a warp moves 512 contiguous bytes
                const float4 *src0 = stop >= 0 ? reinterpret_cast<const float4 *>(fa.incl + (u.unit - (c - stop)) * ustride) + m
                                               : reinterpret_cast<const float4 *>(init);
                const int sq = stop >= 0 ? kRows : 1;
                if (src0) {
#pragma unroll
                    for (int q = 0; q < NS / 4; ++q) {
                        const float4 vv = __ldcg(src0 + q * sq);
                        acc[4 * q] = vv.x;
                        acc[4 * q + 1] = vv.y;
                        acc[4 * q + 2] = vv.z;
                        acc[4 * q + 3] = vv.w;
                    }
                }
                for (int k = stop + 1; k < c; ++k) {
                    const size_t uk = u.unit - (c - k);
                    const float a = __ldcg(fa.alpha + uk * 2 + hh_m);
                    const float4 *src = reinterpret_cast<const float4 *>(fa.agg + uk * ustride) + m;
#pragma unroll
                    for (int q = 0; q < NS / 4; ++q) {
                        const float4 vv = __ldcg(src + q * kRows);
                        acc[4 * q] = fmaf(a, acc[4 * q], vv.x);
                        acc[4 * q + 1] = fmaf(a, acc[4 * q + 1], vv.y);
                        acc[4 * q + 2] = fmaf(a, acc[4 * q + 2], vv.z);
                        acc[4 * q + 3] = fmaf(a, acc[4 * q + 3], vv.w);
                    }
                }
            }
            ok = ok && mbar_wait(&bar_mma[s], ph, lim) && mbar_wait(&bar_seg[ss], pq, lim);
            ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
            tc_fence_after();
            const bool fast = s_fast[ss] != 0;
            // h_{c+1} = a_c h_c + S_c (S_c referenced to the chunk end), 32 columns at a
            // time, stored as it is formed: it is what the successors wait for, so it
            // goes out before the h_c operand of this unit's own off-diagonal product
            if (ok) {
                const float sfac = s_sfac[ss][hh_m], a_own = s_alpha[ss][hh_m];
                float4 *dst = reinterpret_cast<float4 *>(fa.incl + u.unit * ustride) + m;
                const bool wf = unit_is_last<kPacked>(pr, u) && pr.final_state;
#pragma unroll
                for (int cc = 0; cc < NS; cc += 32) {
                    float sc[32];
                    tmem_ld32(slot + col_st + cc, sc);
#pragma unroll
                    for (int k = 0; k < 32; ++k) sc[k] = fmaf(a_own, acc[cc + k], sfac * sc[k]);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 vv = make_float4(sc[4 * q], sc[4 * q + 1], sc[4 * q + 2], sc[4 * q + 3]);
                        __stcg(dst + (cc / 4 + q) * kRows, vv);
                        if (wf)
                            reinterpret_cast<float4 *>(pr.final_state + (((size_t)u.b * H + hg) * P + p_m) * NS)[cc / 4 + q] =
                                vv;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_pincl[s]);  // the team's publisher releases h_{c+1}
            // wx (hi and lo) is dead once the diagonal block's MMAs are done
            ok = ok && mbar_wait(&bar_dg[s], ph, lim);
            if (tt == 0) {  // x of the unit into the staging region (over wx lo): the D x term, and for
                            // a wide unit also the operand of its diagonal block
                if (ok) {
                    mbar_expect_tx(&bar_xe[s], (uint32_t)(2 * kSlab));
                    for (int k = 0; k < 2; ++k)
                        tma_load_3d(st + 2 * kSlab + k * kSlab, &xmap, &bar_xe[s], u.hb * 128 + 64 * k, u.tt, u.tb);
                } else {
                    mbar_arrive(&bar_xe[s]);
                }
            }
            if (ok) {  // e^ref h_c -> bf16 hi / lo K-major slabs over the dead wx hi (ref = 0 in a wide unit)
                const float ysc = s_ysc[ss][hh_m];
#pragma unroll
                for (int q = 0; q < NS / 8; ++q) {
                    float f[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) f[k] = ysc * acc[8 * q + k];
                    uint4 hi, lo;
                    split8(f, hi, lo);
                    *reinterpret_cast<uint4 *>(st + sw128(m, q)) = hi;
                    *reinterpret_cast<uint4 *>(st + kSlab + sw128(m, q)) = lo;
                }
            }
            fence_async_smem();
            tc_fence_before();
            bool any_fail = named_sync_or(bar_team, 128, !ok);
            const uint32_t sbase = tmem + s * 256;
            const uint32_t sa = smem_u32(st);
            const bool row_in = m < u.len;
            uint8_t *ystage = st + 2 * kSlab;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(pr.y) +
                                                   (((size_t)u.tb * pr.seqlen + u.tt + m) * H + u.h0) * P);
            bool okd = !any_fail;
            if (!fast) {
                // A wide unit has no rank-one decay.  Per head, the masked decayed matrix
                // M[m][j] = G_mj e^(cs_m - cs_j) dt_j (j <= m; every factor <= 1 apart from G) is
                // formed in place over G in Y's columns (the diagonal product was skipped) as
                // hi | lo bf16 pairs, 16 columns per 16 tokens, and multiplied with x as loaded
                // (exact in bf16) into S_c's columns (consumed); 64 output columns at a time,
                // each finished in shared memory before the next:
                //   two heads:  Y_off = C h_hh^T in Y's first 64 columns once M_hh is consumed,
                //               y = Y_diag + e^cs Y_off + D x; the next head's M needs G again
                //               (C B^T once more: the stage's B and C are still in place);
                //   one head:   C' = e^cs C (hi, lo over the dead B and over C) joins the same
                //               accumulator, y = (M x + C' h^T) + D x.
                // Each step waits for the MMAs that read what the next one overwrites.
                auto team_sync = [&]() {  // every thread learns whether the leader's steps held
                    tc_fence_before();
                    okd = !named_sync_or(bar_team, 128, !okd);
                    tc_fence_after();
                };
                auto lead_commit_wait = [&]() {
                    mma_commit(&bar_wd[s]);
                    okd = mbar_wait(&bar_wd[s], nwide & 1, lim);
                    ++nwide;
                };
                auto build_m = [&](int hh) {  // M_hh over G, row m = this thread's TMEM lane
                    const float csm = cs[ss][hh * kRows + m];
                    const float *csb = cs[ss] + hh * kRows, *dtb = dtv[ss] + hh * kRows;
#pragma unroll 1
                    for (int jb = 0; jb < 8; ++jb) {
                        uint32_t pk[16];  // 8 hi pairs, then 8 lo pairs
                        if (jb <= 2 * quarter + 1) {  // warp-uniform: some row of this warp reaches 16 jb
                            float gv[16];
                            tmem_ld16(slot + col_y + jb * 16, gv);
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                float f2[2];
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int j = jb * 16 + 2 * k + e;
                                    const float w = __expf(csm - csb[j]) * dtb[j];
                                    f2[e] = j <= m ? gv[2 * k + e] * w : 0.f;
                                }
                                __nv_bfloat162 h2 = __floats2bfloat162_rn(f2[0], f2[1]);
                                const float2 hf = __bfloat1622float2(h2);
                                __nv_bfloat162 l2 = __floats2bfloat162_rn(f2[0] - hf.x, f2[1] - hf.y);
                                pk[k] = *reinterpret_cast<uint32_t *>(&h2);
                                pk[8 + k] = *reinterpret_cast<uint32_t *>(&l2);
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 16; ++k) pk[k] = 0u;
                        }
                        tmem_st16(slot + col_y + jb * 16, pk);
                    }
                };
                // y for the 64 columns `pb` of the unit (x slab pb / 64) from the accumulators
                auto finish64 = [&](int pb, float r, bool with_off, bool last) {
                    const int h = u.h0 + pb / P;
                    const float Dh = pr.D ? __ldg(pr.D + h) : 0.f;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float yd[32], yo[32];
                        tmem_ld32(slot + col_st + 32 * half, yd);
                        if (with_off) tmem_ld32(slot + col_y + 32 * half, yo);
                        if (last && half == 1) {  // this warp's last read of the slot
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bar_slot[s]);
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint4 *sp = reinterpret_cast<uint4 *>(ystage + (pb / 64) * kSlab + sw128(m, 4 * half + k));
                            const uint4 xv = *sp;
                            const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
                            float o[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float2 xf = __bfloat1622float2(x2[e / 2]);
                                const float yoff = with_off ? r * yo[8 * k + e] : 0.f;
                                o[e] = fmaf(Dh, (e & 1) ? xf.y : xf.x, yd[8 * k + e] + yoff);
                            }
                            const uint4 ov = pack8(o);
                            if (tma_out)
                                *sp = ov;
                            else if (row_in)
                                dst[pb / 8 + 4 * half + k] = ov;
                        }
                    }
                };
                const uint32_t id64 = idesc_bf16(128, 64, 0, 1), id64k = idesc_bf16(128, 64, 0, 0);
                // x (staging region) and C are read by every thread below: acquire their loads
                okd = okd && mbar_wait(&bar_xe[s], ph, lim) && mbar_wait(&bar_full[s], ph, lim);
                team_sync();
                if (HB == 2) {
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh > 0 && tt == 0 && okd) {  // G again, over the consumed M and Y_off
                            constexpr uint32_t id_g = idesc_bf16(128, 128, 0, 0);
                            for (int ks = 0; ks < NS / 16; ++ks)
                                mma_bf16(sbase + col_y, sdesc_sw128(sa + 5 * kSlab + ks * 32, 16, 1024),
                                         sdesc_sw128(sa + 4 * kSlab + ks * 32, 16, 1024), id_g, ks > 0);
                            lead_commit_wait();
                        }
                        team_sync();
                        if (okd) build_m(hh);
                        team_sync();
                        if (tt == 0 && okd) {
                            {
                                tc_fence_after();
                                for (int ks = 0; ks < kRows / 16; ++ks) {
                                    const uint64_t xd = sdesc_sw128(sa + 2 * kSlab + hh * kSlab + ks * 2048, kSlab, 1024);
                                    mma_bf16_tA(sbase + col_st, sbase + col_y + 16 * ks, xd, id64, ks > 0);
                                    mma_bf16_tA(sbase + col_st, sbase + col_y + 16 * ks + 8, xd, id64, 1);
                                }
                                lead_commit_wait();
                            }
                            if (okd) {  // Y_off = C h_hh^T (rows 64 hh of the h operand), over M
                                tc_fence_after();
                                for (int ks = 0; ks < NS / 16; ++ks) {
                                    const uint64_t ad = sdesc_sw128(sa + 5 * kSlab + ks * 32, 16, 1024);
                                    mma_bf16(sbase + col_y, ad, sdesc_sw128(sa + hh * 8192 + ks * 32, 16, 1024), id64k,
                                             ks > 0);
                                    mma_bf16(sbase + col_y, ad, sdesc_sw128(sa + kSlab + hh * 8192 + ks * 32, 16, 1024),
                                             id64k, 1);
                                }
                                lead_commit_wait();
                            }
                        }
                        team_sync();
                        if (okd) finish64(64 * hh, rs[ss][hh * kRows + m], true, hh == 1);
                        team_sync();  // the outputs are read before the next head overwrites them
                    }
                } else {
                    if (okd) {
                        build_m(0);
                        // C' = e^cs C for row m: hi over the dead B, lo over C
                        const float ec = rs[ss][m];
#pragma unroll
                        for (int q = 0; q < NS / 8; ++q) {
                            const uint4 cv = *reinterpret_cast<const uint4 *>(st + 5 * kSlab + sw128(m, q));
                            const __nv_bfloat162 *c2 = reinterpret_cast<const __nv_bfloat162 *>(&cv);
                            float f[8];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 cf = __bfloat1622float2(c2[e]);
                                f[2 * e] = ec * cf.x;
                                f[2 * e + 1] = ec * cf.y;
                            }
                            uint4 hi, lo;
                            split8(f, hi, lo);
                            *reinterpret_cast<uint4 *>(st + 4 * kSlab + sw128(m, q)) = hi;
                            *reinterpret_cast<uint4 *>(st + 5 * kSlab + sw128(m, q)) = lo;
                        }
                    }
                    fence_async_smem();
                    team_sync();
                    for (int pb = 0; pb < 128; pb += 64) {
                        if (tt == 0 && okd) {
                            {
                                tc_fence_after();
                                for (int ks = 0; ks < kRows / 16; ++ks) {
                                    const uint64_t xd = sdesc_sw128(sa + 2 * kSlab + (pb / 64) * kSlab + ks * 2048, kSlab, 1024);
                                    mma_bf16_tA(sbase + col_st, sbase + col_y + 16 * ks, xd, id64, ks > 0);
                                    mma_bf16_tA(sbase + col_st, sbase + col_y + 16 * ks + 8, xd, id64, 1);
                                }
                                for (int ks = 0; ks < NS / 16; ++ks) {
                                    const uint64_t chi = sdesc_sw128(sa + 4 * kSlab + ks * 32, 16, 1024);
                                    const uint64_t clo = sdesc_sw128(sa + 5 * kSlab + ks * 32, 16, 1024);
                                    const uint64_t hhi = sdesc_sw128(sa + (pb / 64) * 8192 + ks * 32, 16, 1024);
                                    const uint64_t hlo = sdesc_sw128(sa + kSlab + (pb / 64) * 8192 + ks * 32, 16, 1024);
                                    mma_bf16(sbase + col_st, chi, hhi, id64k, 1);
                                    mma_bf16(sbase + col_st, chi, hlo, id64k, 1);
                                    mma_bf16(sbase + col_st, clo, hhi, id64k, 1);
                                }
                                lead_commit_wait();
                            }
                        }
                        team_sync();
                        if (okd) finish64(pb, 0.f, false, pb == 64);
                        team_sync();  // S_c's columns are read before the next block overwrites them
                    }
                }
                if (tt == 0) {
                    if (okd) mbar_arrive(&bar_free[s]);  // every MMA of the unit is complete
                    mbar_arrive(&bar_yo[s]);
                }
            } else if (tt == 0) {
                // Y += C (e^ref h_c)^T, after the diagonal block's MMAs (issued by another thread,
                // waited for above); the stage's x, B, C are free once it completes
                if (okd) {
                    tc_fence_after();
                    constexpr uint32_t id_o = idesc_bf16(128, 128, 0, 0);
                    for (int ks = 0; ks < NS / 16; ++ks) {
                        const uint64_t ad = sdesc_sw128(sa + 5 * kSlab + ks * 32, 16, 1024);
                        mma_bf16(sbase + col_y, ad, sdesc_sw128(sa + ks * 32, 16, 1024), id_o, 1);
                        mma_bf16(sbase + col_y, ad, sdesc_sw128(sa + kSlab + ks * 32, 16, 1024), id_o, 1);
                    }
                    mma_commit(&bar_yo[s]);
                    mma_commit(&bar_free[s]);
                } else {
                    mbar_arrive(&bar_yo[s]);
                }
            }
            // ---- epilogue of a factored unit: y = r Y + D x, x read from the staging region and
            // y written over it (the same swizzled position), then stored by TMA
            ok = !any_fail && mbar_wait(&bar_yo[s], ph, lim) && mbar_wait(&bar_xe[s], ph, lim);
            ok = __all_sync(0xffffffffu, ok && (fast || okd));  // the TMEM loads below are warp-collective
            tc_fence_after();
            if (ok && fast) {
#pragma unroll
                for (int col = 0; col < 128; col += 64) {
                    const int hh = col / P, h = u.h0 + hh;
                    const float r = rs[ss][hh * kRows + m];
                    const float Dh = pr.D ? __ldg(pr.D + h) : 0.f;
                    float yv[64];
                    tmem_ld64(slot + col_y + col, yv);
                    if (col == 64) {  // this warp's last read of Y: its quarter of the slot is free
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar_slot[s]);
                    }
                    const float2 r2 = make_float2(r, r), D2 = make_float2(Dh, Dh);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint4 *sp = reinterpret_cast<uint4 *>(ystage + (col / 64) * kSlab + sw128(m, k));
                        const uint4 xv = *sp;
                        const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 ry = __fmul2_rn(r2, make_float2(yv[8 * k + 2 * e], yv[8 * k + 2 * e + 1]));
                            const float2 ov2 = __ffma2_rn(D2, __bfloat1622float2(x2[e]), ry);
                            o[2 * e] = ov2.x;
                            o[2 * e + 1] = ov2.y;
                        }
                        const uint4 ov = pack8(o);
                        if (tma_out)
                            *sp = ov;
                        else if (row_in)
                            dst[col / 8 + k] = ov;
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            const bool all_ok = !named_sync_or(bar_team, 128, !ok);
            // every warp frees the slot once per unit: above after its last read, here when it read nothing
            if (!ok && lane == 0) mbar_arrive(&bar_slot[s]);
            if (tt == 0) {
                if (all_ok && tma_out) {
                    for (int k = 0; k < 2; ++k) tma_store_3d(&ymap, ystage + k * kSlab, u.hb * 128 + 64 * k, u.tt, u.tb);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                mbar_arrive(&bar_lo[s]);  // the staging region is free again
            }
            if (!all_ok) {
                s_fail = 1;
                break;
            }
        }
    }
    __syncthreads();
    if (s_fail && tid == 0) atomicOr(pr.err_word, kDevErrTimeout);
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

// [batch][seqlen][width] bf16, 64 x 128 boxes with the 128-byte swizzle
cudaError_t make_map(CUtensorMap *map, const void *ptr, int width, int seqlen, int batch)
{
    return cached_tensor_map(map, ptr, true, width, seqlen, batch, 64, kRows, true);
}

// fp32 [batch][seqlen][width] with a 4 x 128 box (no swizzle), for dt.
cudaError_t make_map_f32(CUtensorMap *map, const void *ptr, int width, int seqlen, int batch)
{
    return cached_tensor_map(map, ptr, false, width, seqlen, batch, 4, kRows, false);
}

// ssd_fused_tc: x | B (then C) | C (then tril(G) hi, then y) | wx ring | h hi/lo | tril(G) lo
size_t fused_smem(int NS)
{
    const size_t body = (size_t)(2 + NS / 64 + 2) * kSlab + 3 * 8192;  // ..., wx ring 24 KiB
    const size_t hreg = NS == 64 ? 0 : (size_t)2 * (NS / 64) * kSlab;
    return 1024 + body + hreg + 2 * kSlab;
}

size_t units_of(const Problem &pr)
{
    const size_t nhb = pr.nheads / (128 / pr.headdim);
    return nhb * (pr.chunks ? (size_t)pr.total_chunks : (size_t)pr.batch * pr.nchunks);
}

template <int NS>
cudaError_t launch(const Problem &pr, const FusedArgs &fa, cudaStream_t s)
{
    CUtensorMap xmap, bmap, cmap, ymap;
    cudaError_t e;
    const int mb = pr.chunks ? 1 : pr.batch;  // packed sequences: one batch row of seqlen tokens
    if ((e = make_map(&xmap, pr.x, pr.nheads * pr.headdim, pr.seqlen, mb)) != cudaSuccess) return e;
    if ((e = make_map(&bmap, pr.B, pr.ngroups * pr.dstate, pr.seqlen, mb)) != cudaSuccess) return e;
    if ((e = make_map(&cmap, pr.C, pr.ngroups * pr.dstate, pr.seqlen, mb)) != cudaSuccess) return e;
    if ((e = make_map(&ymap, pr.y, pr.nheads * pr.headdim, pr.seqlen, mb)) != cudaSuccess) return e;
    const size_t units = units_of(pr);
    if constexpr (NS == 64) {
        const size_t psmem = 1024 + (size_t)2 * kStageBytes + 2 * kDtBytes;
        // dt through TMA when its rows are 16-byte multiples and the base is aligned
        CUtensorMap dtmap;
        memset(&dtmap, 0, sizeof dtmap);
        int dt_tma = (pr.nheads % 4 == 0 && (reinterpret_cast<uintptr_t>(pr.dt) & 15) == 0) ? 1 : 0;
        if (dt_tma && make_map_f32(&dtmap, pr.dt, pr.nheads, pr.seqlen, mb) != cudaSuccess) dt_tma = 0;
        auto kern = pr.chunks ? ssd_fused_pipe_tc<true> : ssd_fused_pipe_tc<false>;
        if ((e = ensure_smem_limit(reinterpret_cast<const void *>(kern), psmem)) != cudaSuccess) return e;
        int nsm = 0;
        if ((e = sm_count(&nsm)) != cudaSuccess) return e;
        const unsigned grid = (unsigned)std::min<size_t>(units, (size_t)nsm);
        if ((e = cudaMemsetAsync(fa.aggcnt, 0, (2 * units + kCtrCount) * sizeof(uint32_t), s)) != cudaSuccess)
            return e;
        profile_kernel_begin(s);
        kern<<<grid, kPipeThreads, psmem, s>>>(xmap, bmap, cmap, ymap, dtmap, pr, fa, (int)units, dt_tma);
        profile_kernel_end(s);
    } else {
        const size_t smem = fused_smem(NS);
        auto kern = pr.chunks ? ssd_fused_tc<NS, true> : ssd_fused_tc<NS, false>;
        if ((e = ensure_smem_limit(reinterpret_cast<const void *>(kern), smem)) != cudaSuccess) return e;
        int nsm = 0;
        if ((e = sm_count(&nsm)) != cudaSuccess) return e;
        const unsigned grid = (unsigned)std::min<size_t>(units, (size_t)nsm);  // one persistent CTA per SM
        if ((e = cudaMemsetAsync(fa.aggcnt, 0, (2 * units + kCtrCount) * sizeof(uint32_t), s)) != cudaSuccess)
            return e;
        profile_kernel_begin(s);
        kern<<<grid, kThreads, smem, s>>>(xmap, bmap, cmap, ymap, pr, fa, (int)units);
        profile_kernel_end(s);
    }
    return cudaGetLastError();
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

bool fused_supported(const Problem &pr)
{
    if (pr.dtype != SSD_DTYPE_BF16) return false;
    if (pr.headdim != 64 && pr.headdim != 128) return false;
    if (pr.dstate != 64 && pr.dstate != 128) return false;
    if (pr.chunk > kRows) return false;
    const int HB = 128 / pr.headdim;
    if (pr.nheads % HB != 0 || (pr.nheads / pr.ngroups) % HB != 0) return false;
    return units_of(pr) < (1u << 31);
}

size_t fused_workspace_bytes(const Problem &pr)
{
    if (seq_supported(pr)) return seq_workspace_bytes(pr);
    const size_t units = units_of(pr);
    const size_t states = units * kRows * pr.dstate * sizeof(float);
    return 2 * up256(states) + up256(units * 2 * sizeof(float)) + up256((2 * units + kCtrCount) * sizeof(uint32_t));
}

cudaError_t launch_fused_tc(const Problem &pr, void *workspace, cudaStream_t s)
{
    if (seq_supported(pr)) return launch_seq_tc(pr, workspace, s);
    const size_t units = units_of(pr);
    const size_t states = units * kRows * pr.dstate * sizeof(float);
    char *p = static_cast<char *>(workspace);
    FusedArgs fa;
    fa.agg = reinterpret_cast<float *>(p);
    p += up256(states);
    fa.incl = reinterpret_cast<float *>(p);
    p += up256(states);
    fa.alpha = reinterpret_cast<float *>(p);
    p += up256(units * 2 * sizeof(float));
    fa.aggcnt = reinterpret_cast<uint32_t *>(p);
    fa.inclcnt = fa.aggcnt + units;
    fa.counters = fa.inclcnt + units;
    return pr.dstate == 64 ? launch<64>(pr, fa, s) : launch<128>(pr, fa, s);
}

}  // namespace ssd
