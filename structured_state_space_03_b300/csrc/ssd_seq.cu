// ssd_seq.cu -- sequence-pipelined bf16 SSD forward on tcgen05 (sm_103a) for
// dstate 64, headdim 64 or 128, chunk <= 128 (ssd_seq_pipe_tc).
//
// Decomposition ("Mamba 模型" §4.1, block decomposition of the semiseparable
// matrix; the algebra is written out in ssd_internal.cuh).  A "sequence" is a
// (batch, head block) pair -- the 128/headdim heads whose (head, headdim) rows
// fill the 128 TMEM lanes -- and a unit is one chunk of one sequence.  Units
// are numbered sequence-major (unit = sequence * nchunks + chunk), and every
// CTA owns a contiguous run of them, fixed on the host: a run is made of
// segments, each the consecutive chunks of one sequence inside the run.  The
// chunk-to-chunk recurrence h_{c+1} = a_c h_c + S_c is carried on chip from one
// chunk of a segment to the next (registers of the state team), so the only
// inter-CTA exchange is at a segment boundary, where a sequence continues on
// the next CTA.  To keep that exchange off the critical path, a CTA whose run
// ends inside a sequence first runs a state-only pass over that last segment
// ("phase 1"): its chunks, last one first, accumulate the segment's aggregate
//     S_seg = sum_{j in seg} exp(sum_{k=j+1..end} dt_k A) dt_j x_j B_j^T
// in one TMEM accumulator (the weights are referenced to the segment end, so
// they never exceed dt_j), and a_seg = exp(sum_seg dt A).  It publishes
// (S_seg, a_seg) at once, then -- once the segment's entry state h_in is known
// (the init state for a segment that starts a sequence, else a look-back over
// the predecessors' publications) -- the end state a_seg h_in + S_seg.  A run's
// first segment, if it continues a sequence, takes its entry state from the
// previous CTA's publication; it is processed after the run's other segments,
// and the last segment (whose entry phase 1 found) first.
// The host balances the runs for one CTA per SM, a phase-1 chunk counting as
// ~0.3 of a full one.
//
// Publication slots (one per CTA) carry a 64-bit flag (tag << 2 | kind) whose
// tag is fresh for every launch, so stale flags never match and the workspace
// needs no clearing.  A CTA waits only on lower-numbered CTAs, which never wait
// on it; every wait is bounded (%globaltimer) and a wait that gives up sets the
// device error word and ends the CTA's roles instead of hanging.
//
// Per chunk ("phase 2"), the arithmetic of the other fused kernels: the
// in-chunk decay is rank one per head with a reference at the midpoint of the
// chunk's cs range, r_i = exp(cs_i - ref), v_j = exp(ref - cs_j), so
//     y_i = r_i [ sum_{j<=i} (C_i . B_j) wx_j + C_i . (e^ref h_c) ] + D x_i,
//     S_c = e^(cs_last - ref) wx^T B,   wx_j = v_j dt_j x_j,
// with one masked tril(C B^T) shared by the heads of the block, and tril, wx and
// e^ref h_c fed to the tensor cores as hi + lo bf16 terms.  A chunk whose cs
// range exceeds 120 (the factors would leave range) keeps the state path with
// the decay referenced to the chunk end and has its outputs formed by the
// epilogue warps from the quadratic form itself: per head the masked decayed
// matrix G_ij exp(cs_i - cs_j) dt_j (every factor <= 1 apart from G) times x on
// the tensor cores, plus exp(cs_i) C_i . h_c.
//
// Warp roles (448 threads, one CTA per SM, all 512 TMEM columns):
//   warp 0       TMA loads of dt, x, B (and C in phase 2) into a free stage
//   warp 1       tcgen05.mma: phase 1 S_seg; phase 2 G = C B^T, S_c and the
//                diagonal block by 16-token slices, the off-diagonal product
//   warps 2-5    front: segment sums, decay factors, tril(G) (hi, lo) into
//                TMEM, D x / r into Y, wx (hi, lo) by slices
//   warps 6-9    state team: the published states of phase 1, the segment
//                entry states, and the chain h_c -> h_{c+1} with the bf16 h
//                operand of each chunk's off-diagonal product
//   warps 10-13  epilogue: y = r Y staged in shared memory and stored by TMA
//                (a wide chunk: x back by TMA, its MMAs issued by the leader)
// Stage s (job j uses s = j & 1), 96 KiB: [0, 32K) x -> wx hi -> h hi | lo;
// [32K, 64K) wx lo -> (x for a wide chunk) -> y; [64K, 80K) B; [80K, 96K) C;
// then 2 KiB of dt per stage.  TMEM slot t (phase-2 job i uses t = i & 1) at
// column 256 t: Y [0,128), S_c [128,192); tril(G) hi [192,256) and lo
// [448,512) serve the job the front and the MMA warp are on (a job's G commit
// follows the previous job's diagonal MMAs from the same thread); phase 1
// accumulates S_seg in slot 1's S_c columns.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <climits>
#include <cstring>
#include <mutex>
#include <vector>

#include "ssd_internal.cuh"
#include "ssd_ptx.cuh"
#include "ssd_tile.cuh"

namespace ssd {
namespace {

using namespace ptx;
using namespace tile;

constexpr int NS = 64;
constexpr int kSeqThreads = 14 * 32;
constexpr int kStageBytes = 6 * kSlab;
constexpr int kDtBytes = kRows * 4 * sizeof(float);  // dt box: 128 tokens x 4 heads
constexpr int kSlices = kRows / 32;  // wx is built, and consumed by the MMAs, 32 tokens at a time
constexpr float kSpanMax = 120.f;
constexpr int kMaxSeqBlocks = 256;
enum { kWLoad = 0, kWMma = 1, kWFront = 2, kWState = 6, kWEpi = 10 };
enum { kBarFront = 1, kBarState = 2, kBarEpi = 3 };
enum : unsigned long long { kKindAgg = 1, kKindIncl = 2 };
// cost of a phase-1 chunk relative to a full one, for balancing the runs
constexpr double kPhase1Cost = 0.3;

struct SeqArgs {
    float *S;                  // [slots][NS/4][128][4] segment aggregates S_seg
    float *H;                  // [slots][NS/4][128][4] segment end states
    float *a;                  // [slots][2] segment decays a_seg per head of the block
    unsigned long long *flag;  // [slots] (tag << 2) | kind
    unsigned long long tag;
    int nblk;
    int bound[kMaxSeqBlocks + 1];  // CTA k owns units [bound[k], bound[k+1])
};

// The job list of one CTA: n1 phase-1 jobs (its last segment, last chunk
// first) when the run ends inside a sequence, then its n2 = hi - lo units in
// phase 2, ordered: the last segment [ls, hi) first (its entry state is the one
// phase 1 found), then whole sequences [mid, ls), then a first segment [lo,
// mid) that continues a sequence (its entry state comes from the previous CTA).
struct Plan {
    int lo, hi, nc, ls, mid, n1, n2, njobs;
};

__device__ __forceinline__ Plan make_plan(const SeqArgs &sa, int nc)
{
    Plan p;
    p.lo = sa.bound[blockIdx.x];
    p.hi = sa.bound[blockIdx.x + 1];
    p.nc = nc;
    p.ls = max(p.lo, (p.hi - 1) / nc * nc);  // first unit of the last segment
    p.mid = (p.lo % nc != 0 && p.ls > p.lo) ? min(p.hi, (p.lo / nc + 1) * nc) : p.lo;
    p.n1 = (p.hi % nc != 0) ? p.hi - p.ls : 0;
    p.n2 = p.hi - p.lo;
    p.njobs = p.n1 + p.n2;
    return p;
}

__device__ __forceinline__ int job_unit(const Plan &p, int j)
{
    if (j < p.n1) return p.hi - 1 - j;
    int k = j - p.n1;
    if (k < p.hi - p.ls) return p.ls + k;
    k -= p.hi - p.ls;
    if (k < p.ls - p.mid) return p.mid + k;
    return p.lo + (k - (p.ls - p.mid));
}

struct Unit {
    int c, b, hb, h0, g, tt, len;
};

__device__ __forceinline__ Unit unit_of(const Problem &pr, int nhb, int unit)
{
    Unit u;
    const int q = unit / pr.nchunks;
    u.c = unit - q * pr.nchunks;
    u.b = q / nhb;
    u.hb = q - u.b * nhb;
    u.h0 = u.hb * (128 / pr.headdim);
    u.g = u.h0 / (pr.nheads / pr.ngroups);
    u.tt = u.c * pr.chunk;
    u.len = min(pr.chunk, pr.seqlen - u.tt);
    return u;
}

// The entry state of a segment whose predecessor segment ends in slot k (state
// team, all 128 threads; row m of the block, head hh_m): walk back to the
// nearest slot with a published end state, every slot in between having
// published its aggregate, and apply h <- a h + S forward from there.  Returns
// false (for every thread) if the walk gave up.
__device__ bool look_back(const SeqArgs &sa, int k, float (&h)[NS], int m, int hh_m, int tt, int lane, uint64_t lim,
                          volatile int *s_walk)
{
    if (tt < 32) {
        int top = k, res = -1;
        const uint64_t t0 = globaltimer();
        for (;;) {
            const int kk = top - lane;
            uint32_t f = 0;  // 0: nothing yet, 1: aggregate, 2: end state
            if (kk >= 0) {
                const unsigned long long v = ld_acquire_u64(sa.flag + kk);
                f = (v >> 2) == sa.tag ? (uint32_t)(v & 3ull) : 0u;
            }
            const uint32_t end_mask = __ballot_sync(0xffffffffu, f == 2u);
            const uint32_t none_mask = __ballot_sync(0xffffffffu, f == 0u);
            const uint32_t newer = end_mask ? (end_mask & (0u - end_mask)) - 1u : 0xffffffffu;
            if ((none_mask & newer) == 0u) {
                if (end_mask) {
                    res = top - (__ffs(end_mask) - 1);
                    break;
                }
                top -= 32;  // 32 aggregates: keep walking
                continue;
            }
            // every lane must take the same exit: the next pass's ballots need all 32
            if (__any_sync(0xffffffffu, globaltimer() - t0 > lim)) break;
            __nanosleep(64);
        }
        if (lane == 0) *s_walk = res;
    }
    named_sync(kBarState, 128);
    const int stop = *s_walk;
    named_sync(kBarState, 128);  // s_walk may be written again by a later walk
    if (stop < 0) return false;
    const float4 *src = reinterpret_cast<const float4 *>(sa.H + (size_t)stop * kRows * NS) + m;
#pragma unroll
    for (int q = 0; q < NS / 4; ++q) {
        const float4 v = __ldcg(src + q * kRows);
        h[4 * q] = v.x;
        h[4 * q + 1] = v.y;
        h[4 * q + 2] = v.z;
        h[4 * q + 3] = v.w;
    }
    for (int kk = stop + 1; kk <= k; ++kk) {
        const float a = __ldcg(sa.a + (size_t)kk * 2 + hh_m);
        const float4 *s4 = reinterpret_cast<const float4 *>(sa.S + (size_t)kk * kRows * NS) + m;
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            const float4 v = __ldcg(s4 + q * kRows);
            h[4 * q] = fmaf(a, h[4 * q], v.x);
            h[4 * q + 1] = fmaf(a, h[4 * q + 1], v.y);
            h[4 * q + 2] = fmaf(a, h[4 * q + 2], v.z);
            h[4 * q + 3] = fmaf(a, h[4 * q + 3], v.w);
        }
    }
    return true;
}

__device__ __forceinline__ void load_init_row(const Problem &pr, int b, int h, int p, float (&hr)[NS])
{
    if (pr.init_state) {
        const float4 *src = reinterpret_cast<const float4 *>(pr.init_state + (((size_t)b * pr.nheads + h) * pr.headdim + p) * NS);
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            const float4 v = __ldg(src + q);
            hr[4 * q] = v.x;
            hr[4 * q + 1] = v.y;
            hr[4 * q + 2] = v.z;
            hr[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < NS; ++k) hr[k] = 0.f;
    }
}

__global__ void __launch_bounds__(kSeqThreads, 1)
    ssd_seq_pipe_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap bmap,
                    const __grid_constant__ CUtensorMap cmap, const __grid_constant__ CUtensorMap ymap,
                    const __grid_constant__ CUtensorMap dtmap, const Problem pr, const __grid_constant__ SeqArgs sa,
                    int dt_tma)
{
    extern __shared__ uint8_t smem_raw[];
    // per stage s: full, dt, free (x region and B, C), lo (wx lo / y staging region), slices;
    // per TMEM slot t: g, mask, mma, hop (h operand written), yo, slot;
    // per phase-2 job (i & 3): seg (the job's scalars written), epi (read by the epilogue);
    // drain: the MMA warp's last commit before the kernel frees TMEM
    __shared__ __align__(8) uint64_t bar_full[2], bar_dt[2], bar_free[2], bar_lo[2], bar_slice[2][kSlices];
    __shared__ __align__(8) uint64_t bar_g[2], bar_mask[2], bar_mma[2], bar_hop[2], bar_yo[2], bar_slot[2];
    __shared__ __align__(8) uint64_t bar_seg[4], bar_epi[4], bar_agg, bar_aggs, bar_aggread, bar_drain;
    // wide jobs: S_c read by the state team (per slot), x back in the staging region, the
    // epilogue leader's MMA steps
    __shared__ __align__(8) uint64_t bar_scr[2], bar_xe, bar_wd;
    __shared__ uint32_t tmem_slot;
    __shared__ float cs[4][2 * kRows], dtv[4][2 * kRows], rs[4][2 * kRows], vwf[2 * kRows];
    __shared__ float s_alpha[4][2], s_sfac[4][2], s_ysc[4][2], s_aseg[2];
    __shared__ float wtot[4][2], wmn[4][2], wmx[4][2];
    __shared__ int s_wide[4];
    __shared__ int s_walk, s_fail;

    const uint64_t lim = pr.wait_ns;  // limit of every bounded wait
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;  // TMEM lane of this thread (warps 2-13)
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int P = pr.headdim, HB = 128 / P, H = pr.nheads, nhb = H / HB, nc = pr.nchunks;
    const Plan pl = make_plan(sa, nc);
    // per slot: Y, S_c; tril(G) hi | lo after each slot's S_c, shared by the jobs (phase 1
    // accumulates S_seg in slot 1's S_c columns)
    constexpr uint32_t col_y = 0, col_st = 128, col_mhi = 192, col_mlo = 448;
    volatile int *vfail = &s_fail;

    if (warp == kWMma) tmem_alloc(&tmem_slot, 512);
    if (tid == 0) {
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bar_full[k], 1);
            mbar_init(&bar_dt[k], 1);
            mbar_init(&bar_free[k], 1);
            mbar_init(&bar_lo[k], 1);
            for (int q = 0; q < kSlices; ++q) mbar_init(&bar_slice[k][q], 128);
            mbar_init(&bar_g[k], 1);
            mbar_init(&bar_mask[k], 128);
            mbar_init(&bar_mma[k], 1);
            mbar_init(&bar_hop[k], 1);
            mbar_init(&bar_yo[k], 1);
            mbar_init(&bar_slot[k], 2);
        }
        for (int k = 0; k < 4; ++k) {
            mbar_init(&bar_seg[k], 128);
            mbar_init(&bar_epi[k], 1);
        }
        mbar_init(&bar_agg, 1);
        mbar_init(&bar_aggs, 128);
        mbar_init(&bar_aggread, 1);
        mbar_init(&bar_drain, 1);
        mbar_init(&bar_scr[0], 1);
        mbar_init(&bar_scr[1], 1);
        mbar_init(&bar_xe, 1);
        mbar_init(&bar_wd, 1);
        mbar_fence_init();
        s_fail = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    uint8_t *base = align1024(smem_raw);
    const float *dt_box = reinterpret_cast<const float *>(base + 2 * kStageBytes);

    if (warp == kWLoad) {
        // ================= TMA loads, one stage per job; the job after next is
        // prefetched into L2 so that its loads, issued once its stage is free,
        // come from L2
        if (lane == 0) {
            tma_prefetch_desc(&xmap);
            tma_prefetch_desc(&bmap);
            tma_prefetch_desc(&cmap);
            if (dt_tma) tma_prefetch_desc(&dtmap);
            auto prefetch = [&](int j) {
                const bool p1 = j < pl.n1;
                const Unit u = unit_of(pr, nhb, job_unit(pl, j));
                if (dt_tma) tma_prefetch_l2_3d(&dtmap, u.h0 & ~3, u.tt, u.b);
                for (int k = 0; k < 2; ++k) tma_prefetch_l2_3d(&xmap, u.hb * 128 + 64 * k, u.tt, u.b);
                tma_prefetch_l2_3d(&bmap, u.g * NS, u.tt, u.b);
                if (!p1) tma_prefetch_l2_3d(&cmap, u.g * NS, u.tt, u.b);
            };
            for (int j = 0; j < 2 && j < pl.njobs; ++j) prefetch(j);
            int last[2] = {-1, -1};  // the last job whose loads went to each stage
            for (int j = 0; j < pl.njobs; ++j) {
                if (*vfail) break;
                const int s = j & 1;
                if (j >= 2 && !mbar_wait(&bar_free[s], ((j >> 1) & 1) ^ 1, lim)) {
                    *vfail = 1;
                    break;
                }
                const bool p1 = j < pl.n1;
                const Unit u = unit_of(pr, nhb, job_unit(pl, j));
                uint8_t *st = base + s * kStageBytes;
                if (dt_tma) {  // dt of the job's 128 tokens x 4 heads from h0 rounded down to 4
                    mbar_expect_tx(&bar_dt[s], (uint32_t)kDtBytes);
                    tma_load_3d(base + 2 * kStageBytes + s * kDtBytes, &dtmap, &bar_dt[s], u.h0 & ~3, u.tt, u.b);
                } else {
                    mbar_arrive(&bar_dt[s]);
                }
                mbar_expect_tx(&bar_full[s], (uint32_t)((p1 ? 3 : 4) * kSlab));
                for (int k = 0; k < 2; ++k)
                    tma_load_3d(st + k * kSlab, &xmap, &bar_full[s], u.hb * 128 + 64 * k, u.tt, u.b);
                tma_load_3d(st + 4 * kSlab, &bmap, &bar_full[s], u.g * NS, u.tt, u.b);
                if (!p1) tma_load_3d(st + 5 * kSlab, &cmap, &bar_full[s], u.g * NS, u.tt, u.b);
                last[s] = j;
                if (j + 2 < pl.njobs) prefetch(j + 2);
            }
            // no copy may still be writing shared memory when the CTA ends (this
            // matters only when a role gave up before consuming its loads)
            for (int s = 0; s < 2; ++s)
                if (last[s] >= 0) {
                    mbar_wait(&bar_dt[s], (last[s] >> 1) & 1, lim);
                    mbar_wait(&bar_full[s], (last[s] >> 1) & 1, lim);
                }
        }
    } else if (warp == kWMma) {
        // ================= tensor-core issue
        if (lane == 0) {
            constexpr uint32_t id_g = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_s = idesc_bf16(128, NS, 1, 1);
            constexpr uint32_t id_d = idesc_bf16(128, 128, 0, 1);
            bool ok = true;
            // Y += C (e^ref h_c)^T for phase-2 job i, the operand being in place
            auto issue_off = [&](int i) {
                const int j = i + pl.n1, s = j & 1, t = i & 1;
                tc_fence_after();
                if (!s_wide[i & 3]) {
                    const uint32_t sa0 = smem_u32(base + s * kStageBytes);
                    for (int ks = 0; ks < NS / 16; ++ks) {
                        const uint64_t ad = sdesc_sw128(sa0 + 5 * kSlab + ks * 32, 16, 1024);
                        mma_bf16(tmem + t * 256 + col_y, ad, sdesc_sw128(sa0 + ks * 32, 16, 1024), id_g, 1);
                        mma_bf16(tmem + t * 256 + col_y, ad, sdesc_sw128(sa0 + kSlab + ks * 32, 16, 1024), id_g, 1);
                    }
                    mma_commit(&bar_yo[t]);
                    mma_commit(&bar_free[s]);
                } else {
                    mbar_arrive(&bar_yo[t]);  // the epilogue frees the stage after its direct evaluation
                }
            };
            for (int j = 0; j < pl.njobs && ok; ++j) {
                if (*vfail) break;
                const int s = j & 1;
                const uint32_t ph = (j >> 1) & 1;
                const uint32_t st = smem_u32(base + s * kStageBytes);
                if (j < pl.n1) {
                    // phase 1: S_seg accumulated in slot 1's chunk-state columns
                    if (!mbar_wait(&bar_full[s], ph, lim)) {
                        ok = false;
                        break;
                    }
                    const uint32_t acc = tmem + 256 + col_st;
                    for (int ks = 0; ks < kSlices && ok; ++ks) {
                        if (!mbar_wait(&bar_slice[s][ks], ph, lim)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        for (int k2 = 2 * ks; k2 < 2 * ks + 2; ++k2) {
                            const uint64_t bd = sdesc_sw128(st + 4 * kSlab + k2 * 2048, kSlab, 1024);
                            mma_bf16(acc, sdesc_sw128(st + k2 * 2048, kSlab, 1024), bd, id_s, (j > 0 || k2 > 0) ? 1u : 0u);
                            mma_bf16(acc, sdesc_sw128(st + 2 * kSlab + k2 * 2048, kSlab, 1024), bd, id_s, 1);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&bar_free[s]);
                    mma_commit(&bar_lo[s]);
                    if (j == pl.n1 - 1) mma_commit(&bar_agg);
                    continue;
                }
                const int i = j - pl.n1, t = i & 1;
                const uint32_t pt = (i >> 1) & 1;
                const uint32_t slot = tmem + t * 256;
                if (i >= 2 && !mbar_wait(&bar_slot[t], pt ^ 1, lim)) {
                    ok = false;
                    break;
                }
                // G = C B^T of this job and the previous job's off-diagonal product,
                // whichever can go first
                bool g_done = false, off_done = i == 0;
                const uint64_t t0 = globaltimer();
                while (!(g_done && off_done)) {
                    if (!g_done && mbar_test_wait(&bar_full[s], ph)) {
                        tc_fence_after();
                        for (int ks = 0; ks < NS / 16; ++ks)
                            mma_bf16(slot + col_y, sdesc_sw128(st + 5 * kSlab + ks * 32, 16, 1024),
                                     sdesc_sw128(st + 4 * kSlab + ks * 32, 16, 1024), id_g, ks > 0);
                        mma_commit(&bar_g[t]);
                        g_done = true;
                    }
                    if (!off_done && mbar_test_wait(&bar_hop[t ^ 1], ((i - 1) >> 1) & 1)) {
                        issue_off(i - 1);
                        off_done = true;
                    }
                    if (!(g_done && off_done) && globaltimer() - t0 > lim) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                // slot 1's chunk-state columns held S_seg until the state team read it
                if (i == 1 && pl.n1 > 0 && !mbar_wait(&bar_aggread, 0, lim)) {
                    ok = false;
                    break;
                }
                // tril(G) and D x / r are in TMEM; then the chunk state and the diagonal
                // block slice by slice as wx arrives (the diagonal block accumulates
                // onto D x / r)
                if (!mbar_wait(&bar_mask[t], pt, lim)) {
                    ok = false;
                    break;
                }
                const bool wide = s_wide[i & 3] != 0;
                for (int ks = 0; ks < kSlices && ok; ++ks) {
                    if (!mbar_wait(&bar_slice[s][ks], ph, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int k2 = 2 * ks; k2 < 2 * ks + 2; ++k2) {
                        const uint64_t bd = sdesc_sw128(st + 4 * kSlab + k2 * 2048, kSlab, 1024);
                        const uint64_t whi = sdesc_sw128(st + k2 * 2048, kSlab, 1024);
                        const uint64_t wlo = sdesc_sw128(st + 2 * kSlab + k2 * 2048, kSlab, 1024);
                        mma_bf16(slot + col_st, whi, bd, id_s, k2 > 0);
                        mma_bf16(slot + col_st, wlo, bd, id_s, 1);
                        if (!wide) {
                            mma_bf16_tA(slot + col_y, tmem + col_mhi + k2 * 8, whi, id_d, 1);
                            mma_bf16_tA(slot + col_y, tmem + col_mhi + k2 * 8, wlo, id_d, 1);
                            mma_bf16_tA(slot + col_y, tmem + col_mlo + k2 * 8, whi, id_d, 1);
                        }
                    }
                }
                if (!ok) break;
                mma_commit(&bar_mma[t]);
            }
            if (ok && !*vfail && pl.n2 > 0) {
                const int i = pl.n2 - 1;
                ok = mbar_wait(&bar_hop[i & 1], (i >> 1) & 1, lim);
                if (ok) issue_off(i);
            }
            if (!ok) *vfail = 1;
            // every MMA issued here (and the arrivals of its commits) is complete
            // before the kernel frees TMEM
            mma_commit(&bar_drain);
            mbar_wait(&bar_drain, 0, lim);
        }
    } else if (warp < kWState) {
        // ================= front: segment sums, factors, tril(G) and D x / r into TMEM, wx slices
        const int ft = tid - 32 * kWFront, fw = warp - kWFront;  // token ft, in warp order
        float Lsuf[2] = {0.f, 0.f};  // phase 1: log-decay from this chunk's end to the segment's end
        for (int j = 0; j < pl.njobs; ++j) {
            if (named_sync_or(kBarFront, 128, *vfail != 0)) break;
            const int s = j & 1;
            const uint32_t ph = (j >> 1) & 1;
            const bool p1 = j < pl.n1;
            const int i = j - pl.n1, t = i & 1, q = i & 3;
            // the epilogue is done with this scalar set (four jobs ago)
            bool ok = p1 || i < 4 || mbar_wait(&bar_epi[q], ((i >> 2) & 1) ^ 1, lim);
            const Unit u = unit_of(pr, nhb, job_unit(pl, j));
            uint8_t *st = base + s * kStageBytes;
            if (dt_tma) ok = ok && mbar_wait(&bar_dt[s], ph, lim);
            const float *dts = dt_box + s * (kDtBytes / 4) + ft * 4 + (u.h0 & 3);
            const size_t trow = (size_t)u.b * pr.seqlen + u.tt + ft;
            float v[2], din[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const bool act = hh < HB && ft < u.len && ok;
                const float a = hh < HB ? __ldg(pr.A + u.h0 + hh) : 0.f;
                const float d = act ? (dt_tma ? dts[hh] : __ldg(pr.dt + trow * H + u.h0 + hh)) : 0.f;
                din[hh] = pr.dtin ? (act ? __ldg(pr.dtin + trow * H + u.h0 + hh) : 0.f) : d;  // input scale
                v[hh] = d * a;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float w = __shfl_up_sync(0xffffffffu, v[hh], o);
                    if (lane >= o) v[hh] += w;
                }
                if (lane == 31) wtot[fw][hh] = v[hh];
            }
            named_sync(kBarFront, 128);
            float tot[2];  // the chunk's sum of dt A (tokens past the chunk end carry 0)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                tot[hh] = (wtot[0][hh] + wtot[1][hh]) + (wtot[2][hh] + wtot[3][hh]);
                for (int w = 0; w < fw; ++w) v[hh] += wtot[w][hh];
            }
            bool fast = true;
            if (p1) {
                // weights referenced to the segment end: exp(sum_{k=j+1..end} dt A) <= 1
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    vwf[hh * kRows + ft] = hh < HB ? expf(Lsuf[hh] + tot[hh] - v[hh]) * din[hh] : 0.f;
                    Lsuf[hh] += tot[hh];
                }
                if (j == pl.n1 - 1) {
                    if (ft < 2) s_aseg[ft] = expf(Lsuf[ft]);
                    mbar_arrive(&bar_aggs);
                }
                named_sync(kBarFront, 128);  // every weight is in shared memory; wtot is free
            } else {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
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
                    cs[q][hh * kRows + ft] = v[hh];
                    dtv[q][hh * kRows + ft] = din[hh];
                }
                named_sync(kBarFront, 128);
                float lo_[2], hi_[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    lo_[hh] = fminf(fminf(wmn[0][hh], wmn[1][hh]), fminf(wmn[2][hh], wmn[3][hh]));
                    hi_[hh] = fmaxf(fmaxf(wmx[0][hh], wmx[1][hh]), fmaxf(wmx[2][hh], wmx[3][hh]));
                }
                fast = (hi_[0] - lo_[0] <= kSpanMax) && (HB == 1 || hi_[1] - lo_[1] <= kSpanMax);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (hh >= HB) break;
                    const float cl = tot[hh];
                    const float ref = 0.5f * (lo_[hh] + hi_[hh]);
                    const float refw = fast ? ref : cl, refy = fast ? ref : 0.f;
                    vwf[hh * kRows + ft] = ft < u.len ? expf(refw - v[hh]) * din[hh] : 0.f;
                    rs[q][hh * kRows + ft] = expf(v[hh] - refy);
                    if (ft == 0) {
                        s_alpha[q][hh] = expf(cl);
                        s_sfac[q][hh] = expf(cl - refw);
                        s_ysc[q][hh] = expf(refy);
                    }
                }
                if (ft == 0) s_wide[q] = fast ? 0 : 1;
                mbar_arrive(&bar_seg[q]);
                named_sync(kBarFront, 128);  // every weight is in shared memory
            }
            ok = ok && mbar_wait(&bar_full[s], ph, lim);
            if (!p1) {
                ok = ok && mbar_wait(&bar_g[t], (i >> 1) & 1, lim);
                ok = __all_sync(0xffffffffu, ok);  // the TMEM accesses below are warp-collective
                tc_fence_after();
                if (ok && fast) {
                    const uint32_t slot = tmem + t * 256 + lane_base;
                    // tril(G) -> hi and lo bf16 pairs (row m) in the shared tril columns; the
                    // previous job's diagonal MMAs, which read them, are complete: this job's G
                    // commit follows them from the same issuing thread
#pragma unroll 1
                    for (int jb = 0; jb < 4; ++jb) {
                        uint32_t ph16[16], pl16[16];
                        if (jb > quarter) {
#pragma unroll
                            for (int k = 0; k < 16; ++k) ph16[k] = pl16[k] = 0u;
                        } else {
                            float gv[32];
                            tmem_ld32(slot + col_y + jb * 32, gv);
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
                    // the Y accumulator starts from D x / r (fp32, token m, every column),
                    // read while x is still in place: y = r Y + D x once the products add up
#pragma unroll 1
                    for (int mb = 0; mb < 2; ++mb) {
                        const int hh = P == 64 ? mb : 0;
                        const float sc = (pr.D ? __ldg(pr.D + u.h0 + hh) : 0.f) / rs[q][hh * kRows + m];
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            uint32_t v16[16];
#pragma unroll
                            for (int c2 = 0; c2 < 2; ++c2) {
                                const uint4 xv = *reinterpret_cast<const uint4 *>(st + mb * kSlab + sw128(m, 2 * kk + c2));
                                const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = __bfloat1622float2(x2[e]);
                                    v16[8 * c2 + 2 * e] = __float_as_uint(f.x * sc);
                                    v16[8 * c2 + 2 * e + 1] = __float_as_uint(f.y * sc);
                                }
                            }
                            tmem_st16(slot + col_y + mb * 64 + 16 * kk, v16);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bar_mask[t]);
                named_sync(kBarFront, 128);  // every x row is read before wx overwrites it
            }
            // the wx lo region of this stage is free again (y of two jobs ago is stored)
            ok = ok && (j < 2 || mbar_wait(&bar_lo[s], ph ^ 1, lim));
            // wx = w dt x: hi in place over x, lo at +32K, in 32-token slices (slice ks
            // is rows 32 ks .. 32 ks + 31 of both 64-column slabs, 512 16-byte chunks)
#pragma unroll 1
            for (int ks = 0; ks < kSlices; ++ks) {
                if (ok) {
                    uint4 xv[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int idx = ft + 128 * r;
                        const int mb = idx >> 8, jr = 32 * ks + ((idx >> 3) & 31), qq = idx & 7;
                        xv[r] = *reinterpret_cast<const uint4 *>(st + mb * kSlab + sw128(jr, qq));
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int idx = ft + 128 * r;
                        const int mb = idx >> 8, jr = 32 * ks + ((idx >> 3) & 31), qq = idx & 7;
                        const float w = vwf[(P == 64 ? mb : 0) * kRows + jr];
                        const __nv_bfloat162 *x2 = reinterpret_cast<const __nv_bfloat162 *>(&xv[r]);
                        const float2 w2 = make_float2(w, w);
                        float f[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 tf = __fmul2_rn(__bfloat1622float2(x2[k]), w2);
                            f[2 * k] = tf.x;
                            f[2 * k + 1] = tf.y;
                        }
                        uint4 hi, lo;
                        split8(f, hi, lo);
                        *reinterpret_cast<uint4 *>(st + mb * kSlab + sw128(jr, qq)) = hi;
                        *reinterpret_cast<uint4 *>(st + 2 * kSlab + mb * kSlab + sw128(jr, qq)) = lo;
                    }
                }
                fence_async_smem();
                mbar_arrive(&bar_slice[s][ks]);
            }
            if (named_sync_or(kBarFront, 128, !ok)) {
                *vfail = 1;
                break;
            }
        }
    } else if (warp < kWEpi) {
        // ================= state team: publications, segment entries, the chain
        const int tt = tid - 32 * kWState;
        const int hh_m = m / P, p_m = m % P;
        const int kslot = blockIdx.x;
        float h[NS];
#pragma unroll
        for (int k = 0; k < NS; ++k) h[k] = 0.f;
        bool ok = true;
        if (pl.n1 > 0) {
            // phase 1: the last segment ends inside its sequence -- publish its
            // aggregate, then its end state a_seg h_in + S_seg
            const Unit u0 = unit_of(pr, nhb, pl.ls);
            const bool head = u0.c == 0;
            const bool withheld = pr.withhold >= pl.ls && pr.withhold < pl.hi;
            ok = mbar_wait(&bar_aggs, 0, lim) && mbar_wait(&bar_agg, 0, lim);
            ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
            tc_fence_after();
            const uint32_t sacc = tmem + 256 + col_st + lane_base;
            if (ok && !head) {
                float4 *dst = reinterpret_cast<float4 *>(sa.S + (size_t)kslot * kRows * NS) + m;
#pragma unroll
                for (int cc = 0; cc < NS; cc += 32) {
                    float sv[32];
                    tmem_ld32(sacc + cc, sv);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcg(dst + (cc / 4 + q) * kRows, make_float4(sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]));
                }
                if (tt < 2) sa.a[(size_t)kslot * 2 + tt] = s_aseg[tt];
            }
            bool fail = named_sync_or(kBarState, 128, !ok);
            if (!fail && !head && tt == 0 && !withheld) st_release_u64(sa.flag + kslot, (sa.tag << 2) | kKindAgg);
            ok = !fail;
            if (ok) {
                if (head)
                    load_init_row(pr, u0.b, u0.h0 + hh_m, p_m, h);
                else
                    ok = look_back(sa, kslot - 1, h, m, hh_m, tt, lane, lim, &s_walk);
            }
            if (ok) {
                const float aseg = s_aseg[hh_m];
                float4 *dst = reinterpret_cast<float4 *>(sa.H + (size_t)kslot * kRows * NS) + m;
#pragma unroll
                for (int cc = 0; cc < NS; cc += 32) {
                    float sv[32];
                    tmem_ld32(sacc + cc, sv);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        __stcg(dst + (cc / 4 + q) * kRows,
                               make_float4(fmaf(aseg, h[cc + 4 * q], sv[4 * q]), fmaf(aseg, h[cc + 4 * q + 1], sv[4 * q + 1]),
                                           fmaf(aseg, h[cc + 4 * q + 2], sv[4 * q + 2]),
                                           fmaf(aseg, h[cc + 4 * q + 3], sv[4 * q + 3])));
                }
            }
            tc_fence_before();
            fail = named_sync_or(kBarState, 128, !ok);
            if (tt == 0) {
                if (!fail && !withheld) st_release_u64(sa.flag + kslot, (sa.tag << 2) | kKindIncl);
                mbar_arrive(&bar_aggread);
            }
            ok = !fail;
        }
        // phase 2: h_c -> operand of chunk c's off-diagonal product -> h_{c+1}
        for (int i = 0; i < pl.n2 && ok; ++i) {
            const int j = i + pl.n1, s = j & 1, t = i & 1, q = i & 3;
            const int unit = job_unit(pl, j);
            const Unit u = unit_of(pr, nhb, unit);
            if (u.c == 0 || unit == pl.lo) {  // a segment starts here
                if (pl.n1 > 0 && unit == pl.ls) {
                    // the last segment: h holds the entry state found in phase 1
                } else if (u.c == 0) {
                    load_init_row(pr, u.b, u.h0 + hh_m, p_m, h);
                } else if (!look_back(sa, kslot - 1, h, m, hh_m, tt, lane, lim, &s_walk)) {
                    ok = false;
                    break;
                }
            }
            ok = mbar_wait(&bar_mma[t], (i >> 1) & 1, lim) && mbar_wait(&bar_seg[q], (i >> 2) & 1, lim);
            tc_fence_after();
            uint8_t *st = base + s * kStageBytes;
            if (ok) {  // e^ref h_c -> bf16 hi / lo K-major slabs over the dead wx hi (ref = 0 if wide)
                const float ysc = s_ysc[q][hh_m];
#pragma unroll
                for (int q8 = 0; q8 < NS / 8; ++q8) {
                    float f[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) f[k] = ysc * h[8 * q8 + k];
                    uint4 hi, lo;
                    split8(f, hi, lo);
                    *reinterpret_cast<uint4 *>(st + sw128(m, q8)) = hi;
                    *reinterpret_cast<uint4 *>(st + kSlab + sw128(m, q8)) = lo;
                }
            }
            fence_async_smem();
            if (named_sync_or(kBarState, 128, !ok)) {
                ok = false;
                break;
            }
            if (tt == 0) mbar_arrive(&bar_hop[t]);
            // h_{c+1} = a_c h_c + S_c (S_c referenced to the chunk end by sfac)
            const float a_own = s_alpha[q][hh_m], sfac = s_sfac[q][hh_m];
            const uint32_t sc_addr = tmem + t * 256 + col_st + lane_base;
#pragma unroll
            for (int cc = 0; cc < NS; cc += 32) {
                float sv[32];
                tmem_ld32(sc_addr + cc, sv);
#pragma unroll
                for (int k = 0; k < 32; ++k) h[cc + k] = fmaf(a_own, h[cc + k], sfac * sv[k]);
            }
            tc_fence_before();
            named_sync(kBarState, 128);
            if (tt == 0) {
                mbar_arrive(&bar_slot[t]);  // S_c read (the epilogue gives the other arrival)
                mbar_arrive(&bar_scr[t]);   // a wide job's epilogue reuses S_c's columns
            }
            if (u.c == nc - 1 && pr.final_state) {
                float4 *fo = reinterpret_cast<float4 *>(pr.final_state +
                                                        (((size_t)u.b * H + u.h0 + hh_m) * P + p_m) * NS);
#pragma unroll
                for (int q4 = 0; q4 < NS / 4; ++q4) fo[q4] = make_float4(h[4 * q4], h[4 * q4 + 1], h[4 * q4 + 2], h[4 * q4 + 3]);
            }
        }
        if (!ok) *vfail = 1;
    } else {
        // ================= epilogue: y = r Y (D x is already in Y), rounded to bf16,
        // staged in the stage's dead wx lo region and stored by TMA
        const int et = tid - 32 * kWEpi;
        // full 128-row tiles go out by TMA (rows past the sequence end are clipped);
        // shorter chunks row by row, since the tile's later rows belong to the next chunk
        const bool tma_out = pr.chunk == kRows;
        int nxe = 0, nwd = 0;  // completed phases of bar_xe and bar_wd (wide jobs only)
        for (int i = 0; i < pl.n2; ++i) {
            if (named_sync_or(kBarEpi, 128, *vfail != 0)) break;
            const int j = i + pl.n1, s = j & 1, t = i & 1, q = i & 3;
            const Unit u = unit_of(pr, nhb, job_unit(pl, j));
            uint8_t *st = base + s * kStageBytes;
            uint8_t *ystage = st + 2 * kSlab;
            bool ok = mbar_wait(&bar_seg[q], (i >> 2) & 1, lim);
            const bool wide = s_wide[q] != 0;
            ok = ok && mbar_wait(&bar_yo[t], (i >> 1) & 1, lim);
            if (wide) ok = ok && mbar_wait(&bar_scr[t], (i >> 1) & 1, lim);
            ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
            tc_fence_after();
            const uint32_t slot = tmem + t * 256 + lane_base;
            const bool row_in = m < u.len;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(pr.y) +
                                                   (((size_t)u.b * pr.seqlen + u.tt + (row_in ? m : 0)) * H + u.h0) * P);
            if (ok && !wide) {
#pragma unroll 1
                for (int col = 0; col < 128; col += 64) {
                    const float r = rs[q][(col / P) * kRows + m];
                    float yv[64];
                    tmem_ld64(slot + col_y + col, yv);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = r * yv[8 * k + e];
                        const uint4 ov = pack8(o);
                        if (tma_out)
                            *reinterpret_cast<uint4 *>(ystage + (col / 64) * kSlab + sw128(m, k)) = ov;
                        else if (row_in)
                            dst[col / 8 + k] = ov;
                    }
                }
            }
            if (wide) {
                // A wide job has no rank-one decay (its outputs are not in Y: the diagonal
                // product was skipped and G = C B^T is still in Y's columns).  Per head, the
                // masked decayed matrix M[m][j] = G_mj e^(cs_m - cs_j) dt_j (j <= m; every factor
                // <= 1 apart from G) is formed in place over G as hi | lo bf16 pairs (16 columns
                // per 16 tokens) and multiplied with x, brought back into the staging region by
                // TMA (exact in bf16), into S_c's columns (read by the state team); 64 output
                // columns at a time, each finished in shared memory before the next:
                //   two heads:  Y_off = C h_hh^T in Y's first 64 columns once M_hh is consumed,
                //               y = Y_diag + e^cs Y_off + D x; the next head's M needs G again
                //               (C B^T once more: the stage's B and C are still in place);
                //   one head:   C' = e^cs C (hi, lo over the dead B and over C) joins the same
                //               accumulator, y = (M x + C' h^T) + D x.
                // The h operand (e^0 h_c, hi and lo) is the state team's.  The leader (et == 0)
                // issues the MMAs and waits for each step before the next overwrites its inputs.
                const uint32_t sbase = tmem + t * 256;
                const uint32_t sa = smem_u32(st);
                bool okd = ok;
                auto team_sync = [&]() {
                    tc_fence_before();
                    okd = !named_sync_or(kBarEpi, 128, !okd);
                    tc_fence_after();
                };
                auto lead_commit_wait = [&]() {
                    mma_commit(&bar_wd);
                    okd = mbar_wait(&bar_wd, nwd & 1, lim);
                    ++nwd;
                };
                team_sync();
                if (et == 0) {  // x into the staging region (wx lo is dead: the chunk state is complete)
                    if (okd) {
                        mbar_expect_tx(&bar_xe, (uint32_t)(2 * kSlab));
                        for (int k = 0; k < 2; ++k)
                            tma_load_3d(ystage + k * kSlab, &xmap, &bar_xe, u.hb * 128 + 64 * k, u.tt, u.b);
                    } else {
                        mbar_arrive(&bar_xe);
                    }
                }
                // x and C are read by every thread below: acquire their loads
                okd = mbar_wait(&bar_xe, nxe & 1, lim) && okd && mbar_wait(&bar_full[s], (j >> 1) & 1, lim);
                ++nxe;
                team_sync();
                auto build_m = [&](int hh) {  // M_hh over G, row m = this thread's TMEM lane
                    const float csm = cs[q][hh * kRows + m];
                    const float *csb = cs[q] + hh * kRows, *dtb = dtv[q] + hh * kRows;
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
                                    const int jj = jb * 16 + 2 * k + e;
                                    const float w = __expf(csm - csb[jj]) * dtb[jj];
                                    f2[e] = jj <= m ? gv[2 * k + e] * w : 0.f;
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
                // y for the 64 columns `pb` of the job (x slab pb / 64) from the accumulators
                auto finish64 = [&](int pb, float r, bool with_off) {
                    const int h = u.h0 + pb / P;
                    const float Dh = pr.D ? __ldg(pr.D + h) : 0.f;
#pragma unroll 1
                    for (int hf = 0; hf < 2; ++hf) {
                        float yd[32], yo[32];
                        tmem_ld32(slot + col_st + 32 * hf, yd);
                        if (with_off) tmem_ld32(slot + col_y + 32 * hf, yo);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint4 *sp = reinterpret_cast<uint4 *>(ystage + (pb / 64) * kSlab + sw128(m, 4 * hf + k));
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
                                dst[pb / 8 + 4 * hf + k] = ov;
                        }
                    }
                };
                const uint32_t id64 = idesc_bf16(128, 64, 0, 1), id64k = idesc_bf16(128, 64, 0, 0);
                if (HB == 2) {
                    for (int hh = 0; hh < 2; ++hh) {
                        if (hh > 0 && et == 0 && okd) {  // G again, over the consumed M and Y_off
                            for (int ks = 0; ks < NS / 16; ++ks)
                                mma_bf16(sbase + col_y, sdesc_sw128(sa + 5 * kSlab + ks * 32, 16, 1024),
                                         sdesc_sw128(sa + 4 * kSlab + ks * 32, 16, 1024), idesc_bf16(128, 128, 0, 0), ks > 0);
                            lead_commit_wait();
                        }
                        team_sync();
                        if (okd) build_m(hh);
                        team_sync();
                        if (et == 0 && okd) {
                            for (int ks = 0; ks < kRows / 16; ++ks) {
                                const uint64_t xd = sdesc_sw128(sa + 2 * kSlab + hh * kSlab + ks * 2048, kSlab, 1024);
                                mma_bf16_tA(sbase + col_st, sbase + col_y + 16 * ks, xd, id64, ks > 0);
                                mma_bf16_tA(sbase + col_st, sbase + col_y + 16 * ks + 8, xd, id64, 1);
                            }
                            lead_commit_wait();
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
                        if (okd) finish64(64 * hh, rs[q][hh * kRows + m], true);
                        team_sync();  // the outputs are read before the next head overwrites them
                    }
                } else {
                    if (okd) {
                        build_m(0);
                        // C' = e^cs C for row m: hi over the dead B, lo over C
                        const float ec = rs[q][m];
#pragma unroll
                        for (int q8 = 0; q8 < NS / 8; ++q8) {
                            const uint4 cv = *reinterpret_cast<const uint4 *>(st + 5 * kSlab + sw128(m, q8));
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
                            *reinterpret_cast<uint4 *>(st + 4 * kSlab + sw128(m, q8)) = hi;
                            *reinterpret_cast<uint4 *>(st + 5 * kSlab + sw128(m, q8)) = lo;
                        }
                    }
                    fence_async_smem();
                    team_sync();
                    for (int pb = 0; pb < 128; pb += 64) {
                        if (et == 0 && okd) {
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
                        team_sync();
                        if (okd) finish64(pb, 0.f, false);
                        team_sync();  // S_c's columns are read before the next block overwrites them
                    }
                }
                if (et == 0 && okd) mbar_arrive(&bar_free[s]);  // every MMA of the job is complete
                ok = okd;
            }
            fence_async_smem();
            tc_fence_before();
            const bool all_ok = !named_sync_or(kBarEpi, 128, !ok);
            if (et == 0) {
                mbar_arrive(&bar_slot[t]);  // Y (and, for a wide job, every column of the slot) read
                mbar_arrive(&bar_epi[q]);   // the job's scalars read
                if (all_ok && tma_out) {
                    for (int k = 0; k < 2; ++k) tma_store_3d(&ymap, ystage + k * kSlab, u.hb * 128 + 64 * k, u.tt, u.b);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                mbar_arrive(&bar_lo[s]);  // the staging region is free again
            }
            if (!all_ok) {
                *vfail = 1;
                break;
            }
        }
        if (et == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // y stores complete
    }
    __syncthreads();
    if (s_fail && tid == 0) atomicOr(pr.err_word, kDevErrTimeout);
    tc_fence_after();
    if (warp == kWMma) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

size_t seq_slots(const Problem &pr)
{
    const size_t units = (size_t)pr.batch * (pr.nheads / (128 / pr.headdim)) * pr.nchunks;
    return std::min<size_t>(units, kMaxSeqBlocks);
}

// Runs of units [bound[k], bound[k+1]) for at most `nblk` CTAs, balanced by a
// cost of 1 per unit plus kPhase1Cost per unit of a run's last segment when
// that segment ends inside its sequence (the chunks of its state-only pass):
// the smallest maximum cost for which a greedy fill needs at most nblk runs.
std::vector<int> make_schedule(int nseq, int nc, int nblk)
{
    const int U = nseq * nc;
    auto cost = [&](int lo, int hi) {
        const int ls = std::max(lo, (hi - 1) / nc * nc);
        const int n1 = hi % nc != 0 ? hi - ls : 0;
        return (double)(hi - lo) + kPhase1Cost * n1;
    };
    auto fill = [&](double T, std::vector<int> *out) {
        int k = 0, lo = 0;
        if (out) out->assign(1, 0);
        while (lo < U) {
            int best = -1;
            for (int hi = lo + 1; hi <= U && (double)(hi - lo) <= T + 1e-9; ++hi)
                if (cost(lo, hi) <= T + 1e-9) best = hi;
            if (best < 0) return INT_MAX;
            lo = best;
            ++k;
            if (out) out->push_back(lo);
        }
        return k;
    };
    double lo_t = (double)U / nblk, hi_t = (double)U * (1.0 + kPhase1Cost) + 1.0;
    for (int it = 0; it < 50 && hi_t - lo_t > 1e-3; ++it) {
        const double mid = 0.5 * (lo_t + hi_t);
        if (fill(mid, nullptr) <= nblk)
            hi_t = mid;
        else
            lo_t = mid;
    }
    std::vector<int> bounds;
    fill(hi_t, &bounds);
    return bounds;
}

struct ScheduleEntry {
    int nseq, nc, nblk;
    std::vector<int> bounds;
};

std::mutex g_sched_mu;
std::vector<ScheduleEntry> g_sched;

std::vector<int> schedule_for(int nseq, int nc, int nblk)
{
    std::lock_guard<std::mutex> lock(g_sched_mu);
    for (const auto &e : g_sched)
        if (e.nseq == nseq && e.nc == nc && e.nblk == nblk) return e.bounds;
    std::vector<int> b = make_schedule(nseq, nc, nblk);
    if (g_sched.size() >= 64) g_sched.erase(g_sched.begin());
    g_sched.push_back({nseq, nc, nblk, b});
    return b;
}

// A fresh 62-bit tag per launch: a flag left in the workspace by an earlier
// launch (or never written) does not carry it.
unsigned long long next_tag()
{
    static std::atomic<unsigned long long> counter{0};
    static const unsigned long long seed = [] {
        const unsigned long long t = (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
        return (t * 0x9E3779B97F4A7C15ull) ^ (reinterpret_cast<uintptr_t>(&counter) << 17);
    }();
    for (;;) {
        const unsigned long long v = (seed + counter.fetch_add(1) * 0xD1B54A32D192ED03ull) & ((1ull << 62) - 1);
        if (v) return v;
    }
}

}  // namespace

// The kernel of choice for few, long sequences.  The persistent look-back kernel
// keeps two units per SM in flight in chunk-major order, so with few (batch,
// head block) sequences most of its units wait on look-back chains a dozen
// chunks deep, while this kernel carries each chain on chip (measured on B300,
// dstate 64, chunk 128: 4 sequences x 512 chunks 155 against 556 us; from ~40
// sequences on, e.g. the 2.7B-shaped layer, the persistent kernel is faster,
// 73 against 92 us).  Pure host decision, no device query.
constexpr int kSeqMaxSequences = 32;

bool seq_supported(const Problem &pr)
{
    const size_t nseq = (size_t)pr.batch * (pr.nheads / (128 / pr.headdim));
    return pr.dstate == NS && !pr.chunks && fused_supported(pr) && nseq <= (size_t)kSeqMaxSequences &&
           nseq * pr.nchunks < (1u << 30);
}

size_t seq_workspace_bytes(const Problem &pr)
{
    const size_t slots = seq_slots(pr);
    return 2 * up256(slots * kRows * NS * sizeof(float)) + up256(slots * 2 * sizeof(float)) +
           up256(slots * sizeof(unsigned long long));
}

cudaError_t launch_seq_tc(const Problem &pr, void *workspace, cudaStream_t s)
{
    CUtensorMap xmap, bmap, cmap, ymap, dtmap;
    cudaError_t e;
    const int W = pr.nheads * pr.headdim, WB = pr.ngroups * pr.dstate;
    if ((e = cached_tensor_map(&xmap, pr.x, true, W, pr.seqlen, pr.batch, 64, kRows, true)) != cudaSuccess) return e;
    if ((e = cached_tensor_map(&bmap, pr.B, true, WB, pr.seqlen, pr.batch, 64, kRows, true)) != cudaSuccess) return e;
    if ((e = cached_tensor_map(&cmap, pr.C, true, WB, pr.seqlen, pr.batch, 64, kRows, true)) != cudaSuccess) return e;
    if ((e = cached_tensor_map(&ymap, pr.y, true, W, pr.seqlen, pr.batch, 64, kRows, true)) != cudaSuccess) return e;
    // dt through TMA when its rows are 16-byte multiples and the base is aligned
    memset(&dtmap, 0, sizeof dtmap);
    int dt_tma = (pr.nheads % 4 == 0 && (reinterpret_cast<uintptr_t>(pr.dt) & 15) == 0) ? 1 : 0;
    if (dt_tma && cached_tensor_map(&dtmap, pr.dt, false, pr.nheads, pr.seqlen, pr.batch, 4, kRows, false) != cudaSuccess)
        dt_tma = 0;
    int nsm = 0;
    if ((e = sm_count(&nsm)) != cudaSuccess) return e;
    const int nseq = pr.batch * (pr.nheads / (128 / pr.headdim));
    const size_t slots = seq_slots(pr);
    const int nblk_max = (int)std::min<size_t>(slots, (size_t)nsm);
    const std::vector<int> bounds = schedule_for(nseq, pr.nchunks, nblk_max);
    SeqArgs sa;
    memset(&sa, 0, sizeof sa);
    char *p = static_cast<char *>(workspace);
    sa.S = reinterpret_cast<float *>(p);
    p += up256(slots * kRows * NS * sizeof(float));
    sa.H = reinterpret_cast<float *>(p);
    p += up256(slots * kRows * NS * sizeof(float));
    sa.a = reinterpret_cast<float *>(p);
    p += up256(slots * 2 * sizeof(float));
    sa.flag = reinterpret_cast<unsigned long long *>(p);
    sa.tag = next_tag();
    sa.nblk = (int)bounds.size() - 1;
    for (size_t k = 0; k < bounds.size(); ++k) sa.bound[k] = bounds[k];
    const size_t smem = 1024 + (size_t)2 * kStageBytes + 2 * kDtBytes;
    if ((e = ensure_smem_limit(reinterpret_cast<const void *>(ssd_seq_pipe_tc), smem)) != cudaSuccess) return e;
    profile_kernel_begin(s);
    ssd_seq_pipe_tc<<<(unsigned)sa.nblk, kSeqThreads, smem, s>>>(xmap, bmap, cmap, ymap, dtmap, pr, sa, dt_tma);
    profile_kernel_end(s);
    return cudaGetLastError();
}

}  // namespace ssd
