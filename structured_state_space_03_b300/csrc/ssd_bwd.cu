// ssd_bwd.cu -- backward of the SSD layer: the gradients of a scalar loss with
// respect to every input, given dL/dy and dL/d(final state).
//
// The pages ask for the intermediate per-token states to be recomputed in the
// backward pass instead of being stored ("Mamba 模型" §3.4, recomputation); here
// nothing of the forward is kept at all.  The same block decomposition as the
// forward ("Mamba 模型" §4.1) is used, with its own chunk length Q = kBQ.  With
// cs_t the in-chunk inclusive prefix of dt A, h_c the state entering chunk c and
// g_c the adjoint of the state leaving it (dL/ds at the chunk's last token from
// every later token; dL/d final state for the last chunk):
//
//   forward chunk states  S_c = sum_j e^{cs_end - cs_j} dt_j x_j B_j^T,
//                         h_{c+1} = e^{cs_end} h_c + S_c,  h_0 = init state
//   adjoint chunk states  G_c = sum_i e^{cs_i} dy_i C_i^T,
//                         g_{c-1} = e^{cs_end} g_c + G_c,  g_last = dfinal,
//                         dinit = g_{-1}
//
// and inside a chunk, with K_ij = e^{cs_i - cs_j} (dy_i . x_j) and
// M_ij = e^{cs_i - cs_j} (C_i . B_j) for i >= j (zero above the diagonal):
//
//   inner_j = sum_i M_ij dy_i + e^{cs_end - cs_j} g_c B_j      (= sum_n B_j[n] dL/ds_j[:, n])
//   dx_j    = D dy_j + dt_j inner_j
//   dB_j    = dt_j (sum_i K_ij C_i + e^{cs_end - cs_j} x_j^T g_c)     (summed over the group's heads)
//   dC_i    = sum_j K_ij dt_j B_j + e^{cs_i} dy_i^T h_c                (summed over the group's heads)
//   dcs_t   = sum_{j<t} W_tj - sum_{i>t} W_it + e^{cs_t} Z_t - e^{cs_end - cs_t} V_t
//             + [t = end] (sum_j e^{cs_end - cs_j} V_j + e^{cs_end} <g_c, h_c>)
//       with W_ij = e^{cs_i - cs_j} (C_i . B_j)(dy_i . x_j) dt_j  (i > j),
//            Z_i = dy_i . (h_c C_i),  V_j = dt_j x_j . (g_c B_j)
//   ddt_u   = x_u . inner_u + A sum_{t >= u} dcs_t,   dA = sum_t dcs_t sum_{u <= t} dt_u,
//   dD      = sum dy . x
//
// Kernels (one CTA per (chunk, head, batch) unless noted; bwd_chunk_tc is persistent):
//   1. chunk states      bf16 / headdim 64 / dstate 64 (128-token chunks): S_c and
//                        the decays by the forward's tcgen05 chunk-state kernel,
//                        then G_c by the same kernel with dy, C and weights e^{cs_j}
//                        (when its head pairs lie inside one group); otherwise
//                        bwd_chunk_states, fp32 FMA (64-token chunks)
//   2. bwd_state_pass    h_c forward and g_c backward over the chunks, dinit
//   3. bwd_chunk_tc      the in-chunk terms on tcgen05 (bf16 / headdim 64 /
//      or bwd_chunk      dstate 64), else on fp32 FMA: dx, ddt, per-head dB / dC,
//                        per-chunk dA / dD parts
//   4. bwd_reduce_*      dB / dC over the heads of a group (when a group has
//                        more than one head), dA / dD over batch and chunks
// Every reduction runs in a fixed order, so results are bitwise reproducible.
#include <algorithm>
#include <cstring>

#include "ssd_internal.cuh"
#include "ssd_ptx.cuh"
#include "ssd_tile.cuh"

namespace ssd {
namespace {

constexpr int kBQ = 64;       // tokens per backward chunk
constexpr int kNS = 32;       // state columns per slice of bwd_chunk
constexpr int kNT = 64;       // state columns per pass of bwd_chunk_states
constexpr int kThreads = 256;

struct BwdArgs {
    const void *x;
    const float *dt;
    const float *A;
    const void *B;
    const void *C;
    const float *D;           // may be null (0)
    const float *init_state;  // may be null (0)
    const void *dy;
    const float *dfinal;      // may be null (0)
    float *dx, *ddt, *dA, *dB, *dC;
    float *dD;                // may be null (not written)
    float *dinit;             // may be null (not written)
    int batch, seqlen, nheads, headdim, ngroups, dstate, nchunks;
    float *hs;                // [b][H][nc][P][N]: S_c, then h_c
    float *gs;                // [b][H][nc][P][N]: G_c, then g_c
    float *decay;             // [b][H][nc]
    float *dBp, *dCp;         // [b][L][H][N] per-head parts (null when one head per group)
    float *dAp, *dDp;         // [b][nc][H] per-chunk parts
    unsigned int *err_word;   // device error word
};

// In-chunk prefix sums of dt*A (cs) and dt (cum) for the Q tokens from t0.
template <int Q>
__device__ __forceinline__ void chunk_scalars(const BwdArgs &a, int b, int h, int t0, int len, float *cs_s,
                                              float *dt_s, float *cum_s, float *warp_tot)
{
    const int tid = threadIdx.x;
    float dtv = 0.f;
    if (tid < len) dtv = __ldg(a.dt + ((size_t)b * a.seqlen + t0 + tid) * a.nheads + h);
    const float cs = block_inclusive_scan_256(dtv * __ldg(a.A + h), warp_tot);
    const float cum = block_inclusive_scan_256(dtv, warp_tot);
    if (tid < Q) {
        cs_s[tid] = cs;
        dt_s[tid] = dtv;
        cum_s[tid] = cum;
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// 1. S_c[p][n] = sum_j e^{cs_end - cs_j} dt_j x_j[p] B_j[n] and
//    G_c[p][n] = sum_i e^{cs_i} dy_i[p] C_i[n], kNT state columns per pass.
//    Thread (ty, tx) owns rows p = ty + 16 a and columns n = tx + 16 q.
template <typename T, int MP, int Q>
__global__ void __launch_bounds__(kThreads) bwd_chunk_states(BwdArgs a)
{
    extern __shared__ float sm[];
    __shared__ float warp_tot[8];
    __shared__ float cs_s[Q], dt_s[Q], cum_s[Q];
    constexpr int PP = MP * 16;
    constexpr int KS = 64;        // tokens staged in shared memory at a time
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int L = a.seqlen, H = a.nheads, P = a.headdim, N = a.dstate, G = a.ngroups;
    const int g = h / (H / G);
    const int t0 = c * Q, len = min(Q, L - t0);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float *xs = sm;               // [KS][PP]  x_j e^{cs_end - cs_j} dt_j
    float *ys = xs + KS * PP;     // [KS][PP]  dy_i e^{cs_i}
    float *bs = ys + KS * PP;     // [KS][kNT]
    float *cm = bs + KS * kNT;    // [KS][kNT]
    const T *x = static_cast<const T *>(a.x);
    const T *dy = static_cast<const T *>(a.dy);
    const T *Bm = static_cast<const T *>(a.B);
    const T *Cm = static_cast<const T *>(a.C);

    chunk_scalars<Q>(a, b, h, t0, len, cs_s, dt_s, cum_s, warp_tot);
    const float cs_end = cs_s[len - 1];
    const size_t bh = (size_t)b * H + h;
    if (tid == 0) a.decay[bh * a.nchunks + c] = expf(cs_end);
    float *S = a.hs + (bh * a.nchunks + c) * (size_t)P * N;
    float *Gc = a.gs + (bh * a.nchunks + c) * (size_t)P * N;
    for (int n0 = 0; n0 < N; n0 += kNT) {
        float accS[MP][4], accG[MP][4];
#pragma unroll
        for (int i = 0; i < MP; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) accS[i][q] = accG[i][q] = 0.f;
        for (int k0 = 0; k0 < len; k0 += KS) {
            const int kn = min(KS, len - k0);
            __syncthreads();  // the previous block's readers are done
            // with one block per chunk, x and dy are staged once for every state-column pass
            if (Q > KS || n0 == 0)
            for (int e = tid; e < KS * PP; e += kThreads) {
                const int t = e / PP, p = e - t * PP;
                float xv = 0.f, yv = 0.f;
                if (t < kn && p < P) {
                    const int tc = k0 + t;
                    const size_t i = (((size_t)b * L + t0 + tc) * H + h) * P + p;
                    xv = load_el(x, i) * (expf(cs_end - cs_s[tc]) * dt_s[tc]);
                    yv = load_el(dy, i) * expf(cs_s[tc]);
                }
                xs[e] = xv;
                ys[e] = yv;
            }
            for (int e = tid; e < KS * kNT; e += kThreads) {
                const int t = e / kNT, n = n0 + (e - t * kNT);
                float bv = 0.f, cv = 0.f;
                if (t < kn && n < N) {
                    const size_t i = (((size_t)b * L + t0 + k0 + t) * G + g) * N + n;
                    bv = load_el(Bm, i);
                    cv = load_el(Cm, i);
                }
                bs[e] = bv;
                cm[e] = cv;
            }
            __syncthreads();
            for (int t = 0; t < kn; ++t) {
                float xv[MP], yv[MP], bv[4], cv[4];
#pragma unroll
                for (int i = 0; i < MP; ++i) {
                    xv[i] = xs[t * PP + ty + 16 * i];
                    yv[i] = ys[t * PP + ty + 16 * i];
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    bv[q] = bs[t * kNT + tx + 16 * q];
                    cv[q] = cm[t * kNT + tx + 16 * q];
                }
#pragma unroll
                for (int i = 0; i < MP; ++i)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        accS[i][q] = fmaf(xv[i], bv[q], accS[i][q]);
                        accG[i][q] = fmaf(yv[i], cv[q], accG[i][q]);
                    }
            }
        }
#pragma unroll
        for (int i = 0; i < MP; ++i) {
            const int p = ty + 16 * i;
            if (p >= P) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = n0 + tx + 16 * q;
                if (n < N) {
                    S[(size_t)p * N + n] = accS[i][q];
                    Gc[(size_t)p * N + n] = accG[i][q];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 2. One thread per (batch, head, state element): h_c forward (S_c -> h_c in
//    place), then g_c backward (G_c -> g_c in place) and dinit = g_{-1}.
__global__ void __launch_bounds__(kThreads) bwd_state_pass(BwdArgs a)
{
    const size_t PN = (size_t)a.headdim * a.dstate;
    const size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (e >= PN) return;
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t bh = (size_t)b * a.nheads + h;
    const int nc = a.nchunks;
    const float *dec = a.decay + bh * nc;
    float *hs = a.hs + bh * nc * PN + e;
    float *gs = a.gs + bh * nc * PN + e;
    // Both sweeps take the chunk states in double-buffered batches of kAhead: the next
    // batch's loads go out before the current batch is applied, so each thread keeps
    // kAhead loads in flight (as the forward's state pass does).
    constexpr int kAhead = 8;
    float s = a.init_state ? a.init_state[bh * PN + e] : 0.f;
    {
        float sc[kAhead], sn[kAhead];
#pragma unroll
        for (int k = 0; k < kAhead; ++k)
            if (k < nc) sc[k] = hs[(size_t)k * PN];
        for (int c0 = 0; c0 < nc; c0 += kAhead) {
#pragma unroll
            for (int k = 0; k < kAhead; ++k)
                if (c0 + kAhead + k < nc) sn[k] = hs[(size_t)(c0 + kAhead + k) * PN];
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                const int c = c0 + k;
                if (c < nc) {
                    hs[(size_t)c * PN] = s;
                    s = fmaf(dec[c], s, sc[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < kAhead; ++k) sc[k] = sn[k];
        }
    }
    float gv = a.dfinal ? a.dfinal[bh * PN + e] : 0.f;
    {
        float sc[kAhead], sn[kAhead];  // k-th entry: chunk nc - 1 - (c0 + k)
#pragma unroll
        for (int k = 0; k < kAhead; ++k)
            if (k < nc) sc[k] = gs[(size_t)(nc - 1 - k) * PN];
        for (int c0 = 0; c0 < nc; c0 += kAhead) {
#pragma unroll
            for (int k = 0; k < kAhead; ++k)
                if (c0 + kAhead + k < nc) sn[k] = gs[(size_t)(nc - 1 - (c0 + kAhead + k)) * PN];
#pragma unroll
            for (int k = 0; k < kAhead; ++k) {
                const int c = nc - 1 - (c0 + k);
                if (c0 + k < nc) {
                    gs[(size_t)c * PN] = gv;
                    gv = fmaf(dec[c], gv, sc[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < kAhead; ++k) sc[k] = sn[k];
        }
    }
    if (a.dinit) a.dinit[bh * PN + e] = gv;
}

// ---------------------------------------------------------------------------
// 3. The in-chunk terms.  Thread (ty, tx) owns, in every [kBQ x *] product,
//    rows ty + 16 r (r < 4) and columns tx + 16 q.
template <typename T, int MP>
__global__ void __launch_bounds__(kThreads) bwd_chunk(BwdArgs a)
{
    extern __shared__ float sm[];
    __shared__ float warp_tot[8];
    __shared__ float cs_s[kBQ], dt_s[kBQ], cum_s[kBQ], eS[kBQ], eC[kBQ];
    __shared__ float Z_s[kBQ], V_s[kBQ], ddt_s[kBQ], row_s[kBQ], col_s[kBQ], dcs_s[kBQ];
    __shared__ float red[16], misc[4];
    constexpr int PP = MP * 16;
    constexpr int XP = PP + 1;   // padded row strides (distinct banks for consecutive rows)
    constexpr int QP = kBQ + 1;
    constexpr int SP = kNS + 1;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int L = a.seqlen, H = a.nheads, P = a.headdim, N = a.dstate, G = a.ngroups;
    const int hpg = H / G, g = h / hpg;
    const int t0 = c * kBQ, len = min(kBQ, L - t0);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float *x_s = sm;                 // [kBQ][XP]
    float *dy_s = x_s + kBQ * XP;    // [kBQ][XP]
    float *k_s = dy_s + kBQ * XP;    // [kBQ][QP]   K
    float *m_s = k_s + kBQ * QP;     // [kBQ][QP]   M
    float *b_s = m_s + kBQ * QP;     // [kBQ][SP]   B slice (then W)
    float *c_s = b_s + kBQ * SP;     // [kBQ][SP]   C slice
    float *h_s = c_s + kBQ * SP;     // [PP][SP]    h_c slice
    float *g_s = h_s + PP * SP;      // [PP][SP]    g_c slice
    const T *x = static_cast<const T *>(a.x);
    const T *dy = static_cast<const T *>(a.dy);
    const T *Bm = static_cast<const T *>(a.B);
    const T *Cm = static_cast<const T *>(a.C);
    const size_t bh = (size_t)b * H + h;
    const size_t PN = (size_t)P * N;
    const float *hc = a.hs + (bh * a.nchunks + c) * PN;
    const float *gc = a.gs + (bh * a.nchunks + c) * PN;

    chunk_scalars<kBQ>(a, b, h, t0, len, cs_s, dt_s, cum_s, warp_tot);
    const float cs_end = cs_s[len - 1];
    if (tid < kBQ) {
        eS[tid] = tid < len ? expf(cs_end - cs_s[tid]) : 0.f;
        eC[tid] = tid < len ? expf(cs_s[tid]) : 0.f;
        Z_s[tid] = V_s[tid] = ddt_s[tid] = 0.f;
    }
    for (int e = tid; e < kBQ * PP; e += kThreads) {
        const int t = e / PP, p = e - t * PP;
        float xv = 0.f, yv = 0.f;
        if (t < len && p < P) {
            const size_t i = (((size_t)b * L + t0 + t) * H + h) * P + p;
            xv = load_el(x, i);
            yv = load_el(dy, i);
        }
        x_s[t * XP + p] = xv;
        dy_s[t * XP + p] = yv;
    }
    __syncthreads();

    // K_ij = e^{cs_i - cs_j} (dy_i . x_j), i >= j; the diagonal gives dD's part.
    {
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
        for (int p = 0; p < P; ++p) {
            float yv[4], xv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) yv[r] = dy_s[(ty + 16 * r) * XP + p];
#pragma unroll
            for (int q = 0; q < 4; ++q) xv[q] = x_s[(tx + 16 * q) * XP + p];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = fmaf(yv[r], xv[q], acc[r][q]);
        }
        float diag = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = ty + 16 * r, j = tx + 16 * q;
                if (i == j) diag += acc[r][q];
                k_s[i * QP + j] = (i >= j && i < len) ? expf(cs_s[i] - cs_s[j]) * acc[r][q] : 0.f;
            }
        if (tx == ty) red[tx] = diag;
    }

    float cb[4][4], bg[4][MP];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
#pragma unroll
        for (int q = 0; q < 4; ++q) cb[r][q] = 0.f;
#pragma unroll
        for (int m = 0; m < MP; ++m) bg[r][m] = 0.f;
    }
    float u_acc = 0.f;
    const bool direct = a.dBp == nullptr;
    float *dBo = direct ? a.dB : a.dBp;
    float *dCo = direct ? a.dC : a.dCp;
    const int rowsH = direct ? G : H;  // heads (or groups) per token row of dBo / dCo
    const int slot = direct ? g : h;

    for (int n0 = 0; n0 < N; n0 += kNS) {
        __syncthreads();  // k_s written; the previous slice's readers done
        for (int e = tid; e < kBQ * kNS; e += kThreads) {
            const int t = e / kNS, nn = e - t * kNS, n = n0 + nn;
            float bv = 0.f, cv = 0.f;
            if (t < len && n < N) {
                const size_t i = (((size_t)b * L + t0 + t) * G + g) * N + n;
                bv = load_el(Bm, i);
                cv = load_el(Cm, i);
            }
            b_s[t * SP + nn] = bv;
            c_s[t * SP + nn] = cv;
        }
        for (int e = tid; e < PP * kNS; e += kThreads) {
            const int p = e / kNS, nn = e - p * kNS, n = n0 + nn;
            float hv = 0.f, gv = 0.f;
            if (p < P && n < N) {
                hv = hc[(size_t)p * N + n];
                gv = gc[(size_t)p * N + n];
            }
            h_s[p * SP + nn] = hv;
            g_s[p * SP + nn] = gv;
            u_acc = fmaf(hv, gv, u_acc);
        }
        __syncthreads();

        // C B^T and B g_c^T, accumulated over the slices
        for (int n = 0; n < kNS; ++n) {
            float cv[4], bq[4], br[4], gv[MP];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                cv[r] = c_s[(ty + 16 * r) * SP + n];
                br[r] = b_s[(ty + 16 * r) * SP + n];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) bq[q] = b_s[(tx + 16 * q) * SP + n];
#pragma unroll
            for (int m = 0; m < MP; ++m) gv[m] = g_s[(tx + 16 * m) * SP + n];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int q = 0; q < 4; ++q) cb[r][q] = fmaf(cv[r], bq[q], cb[r][q]);
#pragma unroll
                for (int m = 0; m < MP; ++m) bg[r][m] = fmaf(br[r], gv[m], bg[r][m]);
            }
        }
        // YH = dy h_c and XG = x g_c for this slice (rows ty + 16 r, columns tx + 16 q, q < 2)
        float yh[4][2], xg[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 2; ++q) yh[r][q] = xg[r][q] = 0.f;
        for (int p = 0; p < P; ++p) {
            float yv[4], xv[4], hv[2], gv[2];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                yv[r] = dy_s[(ty + 16 * r) * XP + p];
                xv[r] = x_s[(ty + 16 * r) * XP + p];
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                hv[q] = h_s[p * SP + tx + 16 * q];
                gv[q] = g_s[p * SP + tx + 16 * q];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    yh[r][q] = fmaf(yv[r], hv[q], yh[r][q]);
                    xg[r][q] = fmaf(xv[r], gv[q], xg[r][q]);
                }
        }
        // Z_i += C_i . YH_i and V_j += B_j . XG_j over this slice (16-lane reductions)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = ty + 16 * r;
            float z = 0.f, v = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                z = fmaf(c_s[i * SP + tx + 16 * q], yh[r][q], z);
                v = fmaf(b_s[i * SP + tx + 16 * q], xg[r][q], v);
            }
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) {
                z += __shfl_xor_sync(0xffffffffu, z, o);
                v += __shfl_xor_sync(0xffffffffu, v, o);
            }
            if (tx == 0) {
                Z_s[i] += z;
                V_s[i] += v;
            }
        }
        // dB_j = dt_j (sum_i K_ij C_i + e^{cs_end - cs_j} XG_j);  dC_i = sum_j K_ij dt_j B_j + e^{cs_i} YH_i
        float db[4][2], dc[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 2; ++q) db[r][q] = dc[r][q] = 0.f;
        for (int k = 0; k < len; ++k) {
            float kj[4], ki[4], cv[2], bv[2];
            const float dtk = dt_s[k];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                kj[r] = k_s[k * QP + ty + 16 * r];          // K_{k, j}
                ki[r] = k_s[(ty + 16 * r) * QP + k] * dtk;  // K_{i, k} dt_k
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                cv[q] = c_s[k * SP + tx + 16 * q];
                bv[q] = b_s[k * SP + tx + 16 * q];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    db[r][q] = fmaf(kj[r], cv[q], db[r][q]);
                    dc[r][q] = fmaf(ki[r], bv[q], dc[r][q]);
                }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int t = ty + 16 * r;
            if (t >= len) continue;
            const size_t row = (((size_t)b * L + t0 + t) * rowsH + slot) * N;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int n = n0 + tx + 16 * q;
                if (n >= N) continue;
                dBo[row + n] = dt_s[t] * fmaf(eS[t], xg[r][q], db[r][q]);
                dCo[row + n] = fmaf(eC[t], yh[r][q], dc[r][q]);
            }
        }
    }
    __syncthreads();  // every reader of the slices done; b_s is reused for W

    // M_ij = e^{cs_i - cs_j} (C_i . B_j) and W_ij = M_ij (dy_i . x_j) dt_j, i >= j
    float *w_s = b_s;  // [kBQ][QP] over b_s and c_s (kBQ * QP <= 2 * kBQ * SP)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = ty + 16 * r, j = tx + 16 * q;
            const bool lower = i >= j && i < len;
            const float e = lower ? expf(cs_s[i] - cs_s[j]) : 0.f;
            m_s[i * QP + j] = e * cb[r][q];
            // K_ij already holds e^{cs_i - cs_j} (dy_i . x_j)
            w_s[i * QP + j] = (lower && i != j) ? cb[r][q] * k_s[i * QP + j] * dt_s[j] : 0.f;
        }
    // U = <g_c, h_c> (block reduction in a fixed order)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) u_acc += __shfl_xor_sync(0xffffffffu, u_acc, o);
    if ((tid & 31) == 0) warp_tot[tid >> 5] = u_acc;
    __syncthreads();
    if (tid < kBQ) {
        float rs = 0.f, cl = 0.f;
        for (int j = 0; j < kBQ; ++j) rs += w_s[tid * QP + j];
        for (int i = 0; i < kBQ; ++i) cl += w_s[i * QP + tid];
        row_s[tid] = rs;
        col_s[tid] = cl;
    } else if (tid == kBQ) {
        float u = 0.f, d = 0.f;
        for (int w = 0; w < 8; ++w) u += warp_tot[w];
        for (int w = 0; w < 16; ++w) d += red[w];
        misc[0] = u;
        misc[1] = d;
    }

    // inner_j = sum_i M_ij dy_i + e^{cs_end - cs_j} (B g_c^T)_j; dx; x . inner
    {
        float inner[4][MP];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int m = 0; m < MP; ++m) inner[r][m] = 0.f;
        for (int i = 0; i < len; ++i) {
            float mv[4], yv[MP];
#pragma unroll
            for (int r = 0; r < 4; ++r) mv[r] = m_s[i * QP + ty + 16 * r];
#pragma unroll
            for (int m = 0; m < MP; ++m) yv[m] = dy_s[i * XP + tx + 16 * m];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int m = 0; m < MP; ++m) inner[r][m] = fmaf(mv[r], yv[m], inner[r][m]);
        }
        const float Dh = a.D ? __ldg(a.D + h) : 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int j = ty + 16 * r;
            float xi = 0.f;
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                const int p = tx + 16 * m;
                const float in = fmaf(eS[j], bg[r][m], inner[r][m]);
                xi = fmaf(x_s[j * XP + p], in, xi);
                if (j < len && p < P)
                    a.dx[(((size_t)b * L + t0 + j) * H + h) * P + p] = fmaf(Dh, dy_s[j * XP + p], dt_s[j] * in);
            }
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) xi += __shfl_xor_sync(0xffffffffu, xi, o);
            if (tx == 0) ddt_s[j] = xi;
        }
    }
    __syncthreads();

    // dcs_t, then ddt and the dA / dD parts
    if (tid == 0) {
        float s = 0.f;
        for (int j = 0; j < len; ++j) s = fmaf(eS[j] * dt_s[j], V_s[j], s);
        misc[2] = s + expf(cs_end) * misc[0];
    }
    __syncthreads();
    if (tid < kBQ) {
        const int t = tid;
        float d = 0.f;
        if (t < len) {
            d = row_s[t] - col_s[t] + eC[t] * Z_s[t] - eS[t] * dt_s[t] * V_s[t];
            if (t == len - 1) d += misc[2];
        }
        dcs_s[t] = d;
    }
    __syncthreads();
    if (tid < len) {
        float r = 0.f;
        for (int t = len - 1; t >= tid; --t) r += dcs_s[t];
        a.ddt[((size_t)b * L + t0 + tid) * H + h] = fmaf(__ldg(a.A + h), r, ddt_s[tid]);
    } else if (tid == kBQ) {
        float s = 0.f;
        for (int t = 0; t < len; ++t) s = fmaf(dcs_s[t], cum_s[t], s);
        const size_t o = ((size_t)b * a.nchunks + c) * H + h;
        a.dAp[o] = s;
        a.dDp[o] = misc[1];
    }
}

// ---------------------------------------------------------------------------
// 4a. dB / dC: sum of the per-head parts over the heads of each group.  With dstate a
//     multiple of 4 (and dB, dC 16-byte aligned): four consecutive state columns as
//     float4s, the heads split over four threads (see below).
__global__ void __launch_bounds__(kThreads) bwd_reduce_groups(BwdArgs a)
{
    // kSub threads per four columns, each summing every kSub-th head of the group; the
    // partial sums are then added in shared memory, in a fixed order (results stay bitwise
    // reproducible), so four times as many loads are in flight
    constexpr int kSub = 4, kOut = kThreads / kSub;
    __shared__ float4 pb[kSub][kOut], pc[kSub][kOut];
    const int H = a.nheads, G = a.ngroups, N = a.dstate, hpg = H / G, N4 = N / 4;
    const size_t total = (size_t)a.batch * a.seqlen * G * N4;
    const float4 *dBp = reinterpret_cast<const float4 *>(a.dBp), *dCp = reinterpret_cast<const float4 *>(a.dCp);
    const int sub = threadIdx.x / kOut, o = threadIdx.x % kOut;
    for (size_t e0 = (size_t)blockIdx.x * kOut; e0 < total; e0 += (size_t)gridDim.x * kOut) {  // block-uniform
        const size_t e = e0 + o;
        float4 sb = make_float4(0.f, 0.f, 0.f, 0.f), sc = sb;
        if (e < total) {
            const int n4 = (int)(e % N4);
            const size_t bt_g = e / N4;
            const int g = (int)(bt_g % G);
            const size_t bt = bt_g / G;
            const size_t base = (bt * H + (size_t)g * hpg) * N4 + n4;
            int k = sub;
            for (; k + kSub < hpg; k += 2 * kSub) {  // two heads' loads in flight per thread
                const float4 vb0 = __ldcs(dBp + base + (size_t)k * N4), vc0 = __ldcs(dCp + base + (size_t)k * N4);
                const float4 vb1 = __ldcs(dBp + base + (size_t)(k + kSub) * N4);
                const float4 vc1 = __ldcs(dCp + base + (size_t)(k + kSub) * N4);
                sb.x += vb0.x; sb.y += vb0.y; sb.z += vb0.z; sb.w += vb0.w;
                sc.x += vc0.x; sc.y += vc0.y; sc.z += vc0.z; sc.w += vc0.w;
                sb.x += vb1.x; sb.y += vb1.y; sb.z += vb1.z; sb.w += vb1.w;
                sc.x += vc1.x; sc.y += vc1.y; sc.z += vc1.z; sc.w += vc1.w;
            }
            for (; k < hpg; k += kSub) {
                const float4 vb = __ldcs(dBp + base + (size_t)k * N4), vc = __ldcs(dCp + base + (size_t)k * N4);
                sb.x += vb.x; sb.y += vb.y; sb.z += vb.z; sb.w += vb.w;
                sc.x += vc.x; sc.y += vc.y; sc.z += vc.z; sc.w += vc.w;
            }
        }
        pb[sub][o] = sb;
        pc[sub][o] = sc;
        __syncthreads();
        if (sub == 0 && e < total) {
            float4 tb = pb[0][o], tc = pc[0][o];
#pragma unroll
            for (int q = 1; q < kSub; ++q) {
                tb.x += pb[q][o].x; tb.y += pb[q][o].y; tb.z += pb[q][o].z; tb.w += pb[q][o].w;
                tc.x += pc[q][o].x; tc.y += pc[q][o].y; tc.z += pc[q][o].z; tc.w += pc[q][o].w;
            }
            reinterpret_cast<float4 *>(a.dB)[e] = tb;
            reinterpret_cast<float4 *>(a.dC)[e] = tc;
        }
        __syncthreads();
    }
}

// The same one column at a time (dstate not a multiple of 4, or dB / dC not 16-byte aligned).
__global__ void __launch_bounds__(kThreads) bwd_reduce_groups_n1(BwdArgs a)
{
    const int H = a.nheads, G = a.ngroups, N = a.dstate, hpg = H / G;
    const size_t total = (size_t)a.batch * a.seqlen * G * N;
    for (size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += (size_t)gridDim.x * kThreads) {
        const int n = (int)(e % N);
        const size_t bt_g = e / N;
        const int g = (int)(bt_g % G);
        const size_t bt = bt_g / G;
        const size_t base = (bt * H + (size_t)g * hpg) * N + n;
        float sb = 0.f, sc = 0.f;
        for (int k = 0; k < hpg; ++k) {
            sb += a.dBp[base + (size_t)k * N];
            sc += a.dCp[base + (size_t)k * N];
        }
        a.dB[e] = sb;
        a.dC[e] = sc;
    }
}

// 4b. dA[h], dD[h]: sums of the per-chunk parts over batch and chunks (one CTA per head).
__global__ void __launch_bounds__(kThreads) bwd_reduce_heads(BwdArgs a)
{
    __shared__ float ra[kThreads], rd[kThreads];
    const int h = blockIdx.x, H = a.nheads;
    const size_t n = (size_t)a.batch * a.nchunks;
    float sa = 0.f, sd = 0.f;
    for (size_t k = threadIdx.x; k < n; k += kThreads) {
        sa += a.dAp[k * H + h];
        sd += a.dDp[k * H + h];
    }
    ra[threadIdx.x] = sa;
    rd[threadIdx.x] = sd;
    __syncthreads();
    for (int s = kThreads / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s) {
            ra[threadIdx.x] += ra[threadIdx.x + s];
            rd[threadIdx.x] += rd[threadIdx.x + s];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.dA[h] = ra[0];
        if (a.dD) a.dD[h] = rd[0];
    }
}

// ---------------------------------------------------------------------------
// 3'. The in-chunk terms on tcgen05 tensor cores (bf16 inputs, headdim 64,
//     dstate 64, 128-token chunks): persistent, one CTA of 256 threads per SM
//     taking the (chunk, head, batch) tiles in turn; warps w and w + 4 own token
//     rows 32 (w & 3) .. 32 (w & 3) + 31 of
//     every accumulator (their TMEM lanes) and split its columns.
//     x, dy, B, C arrive by TMA as 128-byte-swizzled [128 tokens][64] bf16
//     tiles.  Exact bf16 products (dy x^T, C B^T) take the inputs as they are;
//     every fp32 operand (h_c, g_c, dt B, K, M) goes in as hi + lo bf16 terms,
//     so each product carries fp32-level accuracy into its fp32 accumulator.
//     TMEM columns: dy x^T [0,128) then K^T C [0,64) and K (dt B) [64,128);
//     C B^T [128,256) then M^T dy [128,192); C h^T [256,320); B g^T [320,384);
//     dy h [384,448); x g [448,512).
namespace tcb {

using namespace ptx;
using tile::sw128;
using tile::split8;

constexpr int kQ = 128, kD = 64;
constexpr int kTc = 256;          // threads: two warps per TMEM lane quarter
constexpr int kTile = kQ * kD * 2;  // one [128][64] bf16 tile: 16 KiB
// shared-memory layout (bytes from the 1024-aligned base)
constexpr int oX = 0, oDY = kTile, oB = 2 * kTile, oC = 3 * kTile;
constexpr int oBh = 4 * kTile, oBl = 5 * kTile;                  // dt B, hi / lo
constexpr int oHh = 6 * kTile, oHl = oHh + kTile / 2;            // h_c [64 p][64 n], hi / lo
constexpr int oGh = 7 * kTile, oGl = oGh + kTile / 2;            // g_c, hi / lo
constexpr int oKh = 8 * kTile, oKl = 10 * kTile;                 // K then M [128 i][2 x 64 j], hi / lo
constexpr int kSmemTc = 12 * kTile + 1024;

__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return sdesc_sw128(a, 16, 1024); }
__device__ __forceinline__ uint64_t mdesc(uint32_t a) { return sdesc_sw128(a, kTile, 1024); }

// Sum of v[k] over the 32 lanes of the warp for every k, scattered: lane l
// returns the sum for k = l (a halving exchange, 31 shuffles).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < off; ++k) {
            const float send = upper ? v[k] : v[k + off];
            const float keep = upper ? v[k + off] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}

// Sum over the 256 threads in a fixed order (warp_tot: 8 floats); every thread gets it.
// Three block sums at once (256 threads), each in sum256's order; red holds 3 x 8 floats.
__device__ __forceinline__ float3 sum3_256(float a, float b, float c, float (*red)[8])
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
        c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = a;
        red[1][threadIdx.x >> 5] = b;
        red[2][threadIdx.x >> 5] = c;
    }
    __syncthreads();
    float r[3];
#pragma unroll
    for (int k = 0; k < 3; ++k)
        r[k] = ((red[k][0] + red[k][1]) + (red[k][2] + red[k][3])) + ((red[k][4] + red[k][5]) + (red[k][6] + red[k][7]));
    __syncthreads();
    return make_float3(r[0], r[1], r[2]);
}

// Inclusive block scan of v (256 threads) together with the block sums of v and of w, in one
// exchange: returns (prefix, total of v, total of w); red holds 3 x 8 floats.
__device__ __forceinline__ float3 scan_sum2_256(float v, float w, float (*red)[8])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (lane == 31) red[0][warp] = v;
    if (lane == 0) red[2][warp] = w;
    __syncthreads();
    if (warp == 0) {
        float x = lane < 8 ? red[0][lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += t;
        }
        if (lane < 8) red[1][lane] = x;  // inclusive prefix of the warp totals
    }
    __syncthreads();
    const float pre = warp > 0 ? v + red[1][warp - 1] : v;
    const float tot = red[1][7];
    const float ws = ((red[2][0] + red[2][1]) + (red[2][2] + red[2][3])) + ((red[2][4] + red[2][5]) + (red[2][6] + red[2][7]));
    __syncthreads();
    return make_float3(pre, tot, ws);
}

// Row t (64 bf16) of a [128][64] swizzled tile, as floats.
__device__ __forceinline__ void load_row(const uint8_t *tilep, int t, float (&f)[64])
{
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint4 u = *reinterpret_cast<const uint4 *>(tilep + sw128(t, q));
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 v = __bfloat1622float2(b2[e]);
            f[8 * q + 2 * e] = v.x;
            f[8 * q + 2 * e + 1] = v.y;
        }
    }
}

// e_ij = exp(cs_i - cs_j) on the causal triangle of the chunk (0 elsewhere), for
// the 32 columns j = 32 jb ...; cs in shared memory, 16-byte aligned, read as float4s.
// __expf (the hardware exponential): its error is of the order of the fp32 segment
// sums' own (|cs| 2^-24 in the exponent); an accurate expf with scalar loads ran
// without instruction-level parallelism.  Masked entries are discarded whatever
// the exponential gives there.
__device__ __forceinline__ void decay_row(const float *cs, int i, int jb, bool row_in, float (&e)[32])
{
    const float ci = cs[i];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 c4 = reinterpret_cast<const float4 *>(cs + 32 * jb)[q];
        const float cj[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int j = 32 * jb + 4 * q + v;
            const float ev = __expf(ci - cj[v]);
            e[4 * q + v] = (row_in && j <= i) ? ev : 0.f;
        }
    }
}

// 32 values of row i as hi / lo bf16 into a [128][2 x 64] operand (columns 32 jb ...).
__device__ __forceinline__ void store_split32(uint8_t *hi_base, uint8_t *lo_base, int i, int jb, const float (&v)[32])
{
    const int slab = jb >> 1, q0 = (jb & 1) * 4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        uint4 hi, lo;
        split8(&v[8 * u], hi, lo);
        *reinterpret_cast<uint4 *>(hi_base + slab * kTile + sw128(i, q0 + u)) = hi;
        *reinterpret_cast<uint4 *>(lo_base + slab * kTile + sw128(i, q0 + u)) = lo;
    }
}

__global__ void __launch_bounds__(kTc, 1)
    bwd_chunk_tc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap dymap,
                 const __grid_constant__ CUtensorMap bmap, const __grid_constant__ CUtensorMap cmap,
                 const __grid_constant__ CUtensorMap dbmap, const __grid_constant__ CUtensorMap dcmap,
                 const __grid_constant__ CUtensorMap dxmap, BwdArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tmem_slot;
    __shared__ float warp_tot[8];
    __shared__ __align__(16) float cs_s[kQ];  // read as float4s (decay_row)
    __shared__ __align__(16) float dt_s[kQ];  // read as float4s below
    __shared__ float cum_s[kQ], z_s[kQ], zv_s[kQ], ddt_s[kQ];
    __shared__ float row_s[2][kQ], diag_s[2][kQ];
    __shared__ float colp[4][kQ];
    __shared__ float red_s[3][8];
    __shared__ int s_fail;

    const int L = a.seqlen, H = a.nheads, G = a.ngroups;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warps w and w + 4 share TMEM lanes 32 (w & 3) .. (token rows i) and split the columns
    const int quarter = warp & 3, half = warp >> 2;
    const int i = quarter * 32 + lane;
    uint8_t *base = tile::align1024(smem_raw);
    const uint32_t sb = smem_u32(base);

    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        mbar_fence_init();
        s_fail = 0;
    }
    if (warp == 0) tmem_alloc(&tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t lrow = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lanes

    // Persistent: the CTAs take the (chunk, head, batch) tiles in turn, chunk fastest.  Per
    // tile bar_ld completes once and bar_mma three times; the tile count gives the parities.
    const int ntiles = a.nchunks * H * a.batch;
    for (int tile_i = blockIdx.x, k = 0; tile_i < ntiles; tile_i += gridDim.x, ++k) {
        const uint32_t pl = (uint32_t)k & 1u, pm = (uint32_t)(3 * k) & 1u;  // first completion parities
        const int c = tile_i % a.nchunks, h = (tile_i / a.nchunks) % H, b = tile_i / (a.nchunks * H);
        const int g = h / (H / G);
        const int t0 = c * kQ, len = min(kQ, L - t0);
        const size_t bh = (size_t)b * H + h;
        const float *hc = a.hs + (bh * a.nchunks + c) * (size_t)(kD * kD);
        const float *gc = a.gs + (bh * a.nchunks + c) * (size_t)(kD * kD);
        const float Ah = __ldg(a.A + h);

        if (tid == 0) {
            // this chunk's h_c and g_c (16 KiB each, fresh from the state pass) into L2 while the
            // chunk scalars are formed
            bulk_prefetch_l2(hc, (uint32_t)(kD * kD * sizeof(float)));
            bulk_prefetch_l2(gc, (uint32_t)(kD * kD * sizeof(float)));
            tma_prefetch_desc(&xmap);
            tma_prefetch_desc(&dymap);
            tma_prefetch_desc(&bmap);
            tma_prefetch_desc(&cmap);
            mbar_expect_tx(&bar_ld, (uint32_t)(4 * kTile));
            tma_load_3d(base + oX, &xmap, &bar_ld, h * kD, t0, b);
            tma_load_3d(base + oDY, &dymap, &bar_ld, h * kD, t0, b);
            tma_load_3d(base + oB, &bmap, &bar_ld, g * kD, t0, b);
            tma_load_3d(base + oC, &cmap, &bar_ld, g * kD, t0, b);
        }

        // scalars of the chunk (threads 0..127 = tokens): cs (prefix of dt A), dt, cum (prefix of dt)
        {
            const float d = tid < len ? __ldg(a.dt + ((size_t)b * L + t0 + tid) * H + h) : 0.f;
            const float cs_t = block_inclusive_scan_256(d * Ah, warp_tot);
            const float cum_t = block_inclusive_scan_256(d, warp_tot);
            if (tid < kQ) {
                cs_s[tid] = cs_t;
                dt_s[tid] = d;
                cum_s[tid] = cum_t;
            }
        }

        // h_c, g_c -> [64 p][64 n] hi / lo tiles (row p = tid / 4, two 8-column chunks); <g_c, h_c>
        float u = 0.f;
        {
            const int p = tid >> 2, q0 = (tid & 3) * 2;
#pragma unroll
            for (int q = q0; q < q0 + 2; ++q) {
                float hv[8], gv[8];
                const float4 *hp = reinterpret_cast<const float4 *>(hc + p * kD + 8 * q);
                const float4 *gp = reinterpret_cast<const float4 *>(gc + p * kD + 8 * q);
                const float4 h0 = __ldcg(hp), h1 = __ldcg(hp + 1), g0 = __ldcg(gp), g1 = __ldcg(gp + 1);
                hv[0] = h0.x; hv[1] = h0.y; hv[2] = h0.z; hv[3] = h0.w; hv[4] = h1.x; hv[5] = h1.y; hv[6] = h1.z; hv[7] = h1.w;
                gv[0] = g0.x; gv[1] = g0.y; gv[2] = g0.z; gv[3] = g0.w; gv[4] = g1.x; gv[5] = g1.y; gv[6] = g1.z; gv[7] = g1.w;
#pragma unroll
                for (int k = 0; k < 8; ++k) u = fmaf(hv[k], gv[k], u);
                uint4 hi, lo;
                split8(hv, hi, lo);
                *reinterpret_cast<uint4 *>(base + oHh + sw128(p, q)) = hi;
                *reinterpret_cast<uint4 *>(base + oHl + sw128(p, q)) = lo;
                split8(gv, hi, lo);
                *reinterpret_cast<uint4 *>(base + oGh + sw128(p, q)) = hi;
                *reinterpret_cast<uint4 *>(base + oGl + sw128(p, q)) = lo;
            }
        }
        __syncthreads();  // the scalars are in shared memory
        const float dti = dt_s[i];
        bool ok = mbar_wait(&bar_ld, pl);
        // dt_j B_j -> hi / lo (row i, the four 8-column chunks of this half)
        if (ok) {
#pragma unroll
            for (int q = 4 * half; q < 4 * half + 4; ++q) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(base + oB + sw128(i, q));
                const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
                float v[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(b2[e]);
                    v[2 * e] = dti * f.x;
                    v[2 * e + 1] = dti * f.y;
                }
                uint4 hi, lo;
                split8(v, hi, lo);
                *reinterpret_cast<uint4 *>(base + oBh + sw128(i, q)) = hi;
                *reinterpret_cast<uint4 *>(base + oBl + sw128(i, q)) = lo;
            }
        } else {
            s_fail = 1;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        ok = !s_fail;

        // dy x^T, C B^T, C h^T, B g^T, dy h, x g
        if (tid == 0 && ok) {
            tc_fence_after();
            constexpr uint32_t id_sq = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t id_kk = idesc_bf16(128, 64, 0, 0);
            constexpr uint32_t id_km = idesc_bf16(128, 64, 0, 1);
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                const uint32_t kk = ks * 32, km = ks * 2048;  // K step: 16 elements of a row / 16 rows
                mma_bf16(tmem + 0, kdesc(sb + oDY + kk), kdesc(sb + oX + kk), id_sq, ks > 0);
                mma_bf16(tmem + 128, kdesc(sb + oC + kk), kdesc(sb + oB + kk), id_sq, ks > 0);
                mma_bf16(tmem + 256, kdesc(sb + oC + kk), kdesc(sb + oHh + kk), id_kk, ks > 0);
                mma_bf16(tmem + 256, kdesc(sb + oC + kk), kdesc(sb + oHl + kk), id_kk, 1);
                mma_bf16(tmem + 320, kdesc(sb + oB + kk), kdesc(sb + oGh + kk), id_kk, ks > 0);
                mma_bf16(tmem + 320, kdesc(sb + oB + kk), kdesc(sb + oGl + kk), id_kk, 1);
                mma_bf16(tmem + 384, kdesc(sb + oDY + kk), mdesc(sb + oHh + km), id_km, ks > 0);
                mma_bf16(tmem + 384, kdesc(sb + oDY + kk), mdesc(sb + oHl + km), id_km, 1);
                mma_bf16(tmem + 448, kdesc(sb + oX + kk), mdesc(sb + oGh + km), id_km, ks > 0);
                mma_bf16(tmem + 448, kdesc(sb + oX + kk), mdesc(sb + oGl + km), id_km, 1);
            }
            mma_commit(&bar_mma);
        }
        ok = ok && mbar_wait(&bar_mma, pm);
        ok = __all_sync(0xffffffffu, ok);  // the TMEM loads below are warp-collective
        tc_fence_after();

        // K = e o (dy x^T) -> hi / lo operand; W = e o (C B^T) o (dy x^T) dt_j below the diagonal:
        // row sums here, column sums by a per-warp exchange; the diagonal of dy x^T gives dD's part.
        // This half: column blocks 2 half, 2 half + 1.
        const bool row_in = i < len;
        {
            float rs = 0.f, diag = 0.f;
            if (ok) {
#pragma unroll 1
                for (int jb = 2 * half; jb < 2 * half + 2; ++jb) {
                    float dx[32], cb[32], e[32], w[32];
                    tmem_ld32(lrow + 32 * jb, dx);
                    tmem_ld32(lrow + 128 + 32 * jb, cb);
                    decay_row(cs_s, i, jb, row_in, e);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 d4 = reinterpret_cast<const float4 *>(dt_s + 32 * jb)[q];
                        const float dj[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int k = 4 * q + v, j = 32 * jb + k;
                            if (j == i) diag = dx[k];
                            const float kv = e[k] * dx[k];
                            w[k] = j < i ? kv * cb[k] * dj[v] : 0.f;
                            rs += w[k];
                            dx[k] = kv;
                        }
                    }
                    store_split32(base + oKh, base + oKl, i, jb, dx);
                    colp[quarter][32 * jb + lane] = reduce_scatter32(w, lane);
                }
            }
            row_s[half][i] = rs;
            diag_s[half][i] = diag;
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();

        // K^T C and K (dt B)
        if (tid == 0 && ok) {
            tc_fence_after();
            constexpr uint32_t id_mm = idesc_bf16(128, 64, 1, 1);
            constexpr uint32_t id_km = idesc_bf16(128, 64, 0, 1);
#pragma unroll
            for (int ks = 0; ks < kQ / 16; ++ks) {
                const uint32_t km = ks * 2048;                                    // 16 rows of a [128][..] operand
                const uint32_t kk = (ks >> 2) * kTile + (ks & 3) * 32;            // 16 columns of the K operand
                mma_bf16(tmem + 0, mdesc(sb + oKh + km), mdesc(sb + oC + km), id_mm, ks > 0);
                mma_bf16(tmem + 0, mdesc(sb + oKl + km), mdesc(sb + oC + km), id_mm, 1);
                mma_bf16(tmem + 64, kdesc(sb + oKh + kk), mdesc(sb + oBh + km), id_km, ks > 0);
                mma_bf16(tmem + 64, kdesc(sb + oKh + kk), mdesc(sb + oBl + km), id_km, 1);
                mma_bf16(tmem + 64, kdesc(sb + oKl + kk), mdesc(sb + oBh + km), id_km, 1);
            }
            mma_commit(&bar_mma);
        }
        // meanwhile, from columns the MMAs above do not touch: Z_i = dy_i . (C_i h^T) (first half),
        // V_i = dt_i x_i . (B_i g^T) (second half)
        if (ok) {
            float r[64], f[64];
            tmem_ld64(lrow + (half == 0 ? 256 : 320), r);
            load_row(base + (half == 0 ? oDY : oX), i, f);
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 64; ++k) acc = fmaf(f[k], r[k], acc);
            if (half == 0)
                z_s[i] = acc;
            else
                zv_s[i] = row_in ? expf(cs_s[len - 1] - cs_s[i]) * dti * acc : 0.f;  // e^{cs_end - cs_i} V_i
        }
        ok = ok && mbar_wait(&bar_mma, pm ^ 1u);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();

        // M = e o (C B^T) -> hi / lo over the K operand, then M^T dy
        if (ok) {
#pragma unroll 1
            for (int jb = 2 * half; jb < 2 * half + 2; ++jb) {
                float cb[32], e[32];
                tmem_ld32(lrow + 128 + 32 * jb, cb);
                decay_row(cs_s, i, jb, row_in, e);
#pragma unroll
                for (int k = 0; k < 32; ++k) cb[k] *= e[k];
                store_split32(base + oKh, base + oKl, i, jb, cb);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {
            tc_fence_after();
            constexpr uint32_t id_mm = idesc_bf16(128, 64, 1, 1);
#pragma unroll
            for (int ks = 0; ks < kQ / 16; ++ks) {
                const uint32_t km = ks * 2048;
                mma_bf16(tmem + 128, mdesc(sb + oKh + km), mdesc(sb + oDY + km), id_mm, ks > 0);
                mma_bf16(tmem + 128, mdesc(sb + oKl + km), mdesc(sb + oDY + km), id_mm, 1);
            }
            mma_commit(&bar_mma);
        }
        ok = ok && mbar_wait(&bar_mma, pm);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();

        // outputs of row i: dB and dC (first half; per head, or the group's when it has one
        // head), dx and x . inner (second half)
        const float cs_end = cs_s[len - 1], cs_i = cs_s[i];
        const float eS = row_in ? expf(cs_end - cs_i) : 0.f, eC = row_in ? expf(cs_i) : 0.f;
        // Each row goes into an fp32 staging tile (dB over B and C, dC over dt B, dx over K: all
        // dead now) of two [128][32] boxes with the 128-byte swizzle, so that a warp's row stores
        // spread over the banks; the boxes then go out by TMA (rows past the sequence end are
        // clipped by the tensor maps; the tensor-core backward has no packed layout).
        uint8_t *stB = base + oB, *stC = base + oBh, *stX = base + oKh;
        auto put_row = [&](uint8_t *tile, const float (&v)[64]) {
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4 *>(tile + hb * kTile + sw128(i, q)) =
                        make_float4(v[32 * hb + 4 * q], v[32 * hb + 4 * q + 1], v[32 * hb + 4 * q + 2],
                                    v[32 * hb + 4 * q + 3]);
        };
        if (ok && half == 0) {
            float acc[64], add[64];
            tmem_ld64(lrow + 0, acc);
            tmem_ld64(lrow + 448, add);
#pragma unroll
            for (int k = 0; k < 64; ++k) acc[k] = dti * fmaf(eS, add[k], acc[k]);
            put_row(stB, acc);
            tmem_ld64(lrow + 64, acc);
            tmem_ld64(lrow + 384, add);
#pragma unroll
            for (int k = 0; k < 64; ++k) acc[k] = fmaf(eC, add[k], acc[k]);
            put_row(stC, acc);
        } else if (ok) {
            float acc[64], add[64], f[64];
            tmem_ld64(lrow + 128, acc);
            tmem_ld64(lrow + 320, add);
            const float Dh = a.D ? __ldg(a.D + h) : 0.f;
#pragma unroll
            for (int k = 0; k < 64; ++k) acc[k] = fmaf(eS, add[k], acc[k]);  // inner_i
            load_row(base + oX, i, f);
            float xin = 0.f;
#pragma unroll
            for (int k = 0; k < 64; ++k) xin = fmaf(f[k], acc[k], xin);
            ddt_s[i] = xin;
            load_row(base + oDY, i, f);
#pragma unroll
            for (int k = 0; k < 64; ++k) acc[k] = fmaf(Dh, f[k], dti * acc[k]);
            put_row(stX, acc);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {
            const bool direct = a.dBp == nullptr;  // one head per group: dB and dC themselves
            for (int hb = 0; hb < 2; ++hb) {
                tma_store_3d(&dbmap, stB + hb * kTile, (direct ? g : h) * kD + 32 * hb, t0, b);
                tma_store_3d(&dcmap, stC + hb * kTile, (direct ? g : h) * kD + 32 * hb, t0, b);
                tma_store_3d(&dxmap, stX + hb * kTile, h * kD + 32 * hb, t0, b);
            }
            bulk_commit();
            bulk_wait_read_all();
        }

        // dL/dcs_t (threads 0..127 = tokens t), then ddt = x . inner + A sum_{t' >= t} dcs_t' and the
        // dA / dD parts; sums over all 256 threads in a fixed order (the second half adds zeros)
        const bool tok = tid < kQ && tid < len;
        const float zv = tok ? zv_s[tid] : 0.f;
        // sum_j e^{cs_end - cs_j} V_j, the u sum and the diagonal sum in one exchange
        const float3 s3 = sum3_256(zv, u, tid < kQ ? diag_s[0][tid] + diag_s[1][tid] : 0.f, red_s);
        const float ssum = s3.x, usum = s3.y, dsum = s3.z;
        float d = 0.f;
        if (tok) {
            const float colsum = (colp[0][tid] + colp[1][tid]) + (colp[2][tid] + colp[3][tid]);
            d = (row_s[0][tid] + row_s[1][tid]) - colsum + expf(cs_s[tid]) * z_s[tid] - zv;
            if (tid == len - 1) d += ssum + expf(cs_end) * usum;
        }
        // the prefix of d, its total and the dA part sum_t d_t cum_t in one exchange
        const float3 pt = scan_sum2_256(d, tid < kQ ? d * cum_s[tid] : 0.f, red_s);
        const float pre = pt.x, tot = pt.y, da = pt.z;
        if (tok && ok) a.ddt[((size_t)b * L + t0 + tid) * H + h] = fmaf(Ah, tot - pre + d, ddt_s[tid]);
        if (tid == 0 && ok) {
            const size_t o = ((size_t)b * a.nchunks + c) * H + h;
            a.dAp[o] = da;
            a.dDp[o] = dsum;
        }
        if (tid == 0 && !ok && a.err_word) atomicOr(a.err_word, kDevErrTimeout);
        if (!ok) s_fail = 1;
        tc_fence_before();
        __syncthreads();  // the tile is done with TMEM and shared memory
        tc_fence_after();
        if (s_fail) break;  // block-uniform: read after the barrier
    }  // tiles
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace tcb

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

template <int MP, int Q>
size_t chunk_states_smem() { return sizeof(float) * (2 * 64 * MP * 16 + 2 * 64 * kNT); }
template <int MP>
size_t chunk_smem() { return sizeof(float) * (2 * kBQ * (MP * 16 + 1) + 2 * kBQ * (kBQ + 1) + 2 * kBQ * (kNS + 1) + 2 * MP * 16 * (kNS + 1)); }

cudaError_t launch_reductions(const BwdArgs &a, cudaStream_t s)
{
    cudaError_t e;
    if (a.dBp) {
        int sms = 148;
        if ((e = sm_count(&sms)) != cudaSuccess) return e;
        const bool v4 = a.dstate % 4 == 0 && reinterpret_cast<uintptr_t>(a.dB) % 16 == 0 &&
                        reinterpret_cast<uintptr_t>(a.dC) % 16 == 0;
        const size_t total = (size_t)a.batch * a.seqlen * a.ngroups * a.dstate / (v4 ? 4 : 1);
        const size_t per_block = v4 ? kThreads / 4 : kThreads;  // outputs per block
        const size_t want = (total + per_block - 1) / per_block;
        const unsigned blocks = (unsigned)std::min<size_t>(want, (size_t)sms * 8);
        profile_kernel_begin(s);
        if (v4)
            bwd_reduce_groups<<<blocks, kThreads, 0, s>>>(a);
        else
            bwd_reduce_groups_n1<<<blocks, kThreads, 0, s>>>(a);
        profile_kernel_end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    profile_kernel_begin(s);
    bwd_reduce_heads<<<a.nheads, kThreads, 0, s>>>(a);
    profile_kernel_end(s);
    return cudaGetLastError();
}

template <typename T, int MP>
cudaError_t launch_bwd_typed(const BwdArgs &a, cudaStream_t s)
{
    const dim3 grid(a.nchunks, a.nheads, a.batch);
    cudaError_t e;
    const size_t s1 = chunk_states_smem<MP, kBQ>(), s3 = chunk_smem<MP>();
    if ((e = ensure_smem_limit((const void *)bwd_chunk_states<T, MP, kBQ>, s1)) != cudaSuccess) return e;
    if ((e = ensure_smem_limit((const void *)bwd_chunk<T, MP>, s3)) != cudaSuccess) return e;
    profile_kernel_begin(s);
    bwd_chunk_states<T, MP, kBQ><<<grid, kThreads, s1, s>>>(a);
    profile_kernel_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t PN = (size_t)a.headdim * a.dstate;
    profile_kernel_begin(s);
    bwd_state_pass<<<dim3((unsigned)((PN + kThreads - 1) / kThreads), a.nheads, a.batch), kThreads, 0, s>>>(a);
    profile_kernel_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    profile_kernel_begin(s);
    bwd_chunk<T, MP><<<grid, kThreads, s3, s>>>(a);
    profile_kernel_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_reductions(a, s);
}

// bf16, headdim 64, dstate 64: chunk states and state passes as on the fp32 path
// (128-token chunks), the in-chunk terms on tcgen05
cudaError_t launch_bwd_tc(const BwdArgs &a, cudaStream_t s)
{
    CUtensorMap xm, dym, bm, cm;
    cudaError_t e;
    const int H = a.nheads, G = a.ngroups;
    if ((e = cached_tensor_map(&xm, a.x, true, H * 64, a.seqlen, a.batch, 64, 128, true)) != cudaSuccess) return e;
    if ((e = cached_tensor_map(&dym, a.dy, true, H * 64, a.seqlen, a.batch, 64, 128, true)) != cudaSuccess) return e;
    if ((e = cached_tensor_map(&bm, a.B, true, G * 64, a.seqlen, a.batch, 64, 128, true)) != cudaSuccess) return e;
    if ((e = cached_tensor_map(&cm, a.C, true, G * 64, a.seqlen, a.batch, 64, 128, true)) != cudaSuccess) return e;
    // fp32 outputs of the in-chunk kernel, stored by TMA from [128][32] swizzled boxes: dB and
    // dC per head (their parts) or per group (one head per group), dx
    CUtensorMap dbm, dcm, dxm;
    const bool parts = a.dBp != nullptr;
    if ((e = cached_tensor_map(&dbm, parts ? a.dBp : a.dB, false, (parts ? H : G) * 64, a.seqlen, a.batch, 32, 128,
                               true)) != cudaSuccess)
        return e;
    if ((e = cached_tensor_map(&dcm, parts ? a.dCp : a.dC, false, (parts ? H : G) * 64, a.seqlen, a.batch, 32, 128,
                               true)) != cudaSuccess)
        return e;
    if ((e = cached_tensor_map(&dxm, a.dx, false, H * 64, a.seqlen, a.batch, 32, 128, true)) != cudaSuccess) return e;
    const dim3 grid(a.nchunks, H, a.batch);
    const size_t s1 = chunk_states_smem<4, tcb::kQ>();
    if (H % 2 == 0 && (H / G) % 2 == 0) {
        // S_c and the chunk decays are exactly the forward's chunk-state product: on
        // tcgen05 (its head pairs lie inside one group); G_c too, with other weights
        Problem fp;
        memset(&fp, 0, sizeof fp);
        fp.x = a.x;
        fp.dt = a.dt;
        fp.A = a.A;
        fp.B = a.B;
        fp.C = a.C;
        fp.batch = a.batch;
        fp.seqlen = a.seqlen;
        fp.nheads = H;
        fp.headdim = 64;
        fp.ngroups = G;
        fp.dstate = 64;
        fp.chunk = tcb::kQ;
        fp.nchunks = a.nchunks;
        fp.dtype = SSD_DTYPE_BF16;
        fp.err_word = a.err_word;
        Workspace fws;
        fws.states = a.hs;
        fws.decay = a.decay;
        if ((e = launch_chunk_state_tc(fp, fws, s)) != cudaSuccess) return e;
        // G_c = sum_i e^{cs_i} dy_i C_i^T: the same product with dy, C and the weights e^{cs_i}
        fp.x = a.dy;
        fp.B = a.C;
        fp.adjoint_states = 1;
        fws.states = a.gs;
        if ((e = launch_chunk_state_tc(fp, fws, s)) != cudaSuccess) return e;
    } else {  // both state sums on the fp32 kernel
        if ((e = ensure_smem_limit((const void *)bwd_chunk_states<__nv_bfloat16, 4, tcb::kQ>, s1)) != cudaSuccess)
            return e;
        profile_kernel_begin(s);
        bwd_chunk_states<__nv_bfloat16, 4, tcb::kQ><<<grid, kThreads, s1, s>>>(a);
        profile_kernel_end(s);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = ensure_smem_limit((const void *)tcb::bwd_chunk_tc, tcb::kSmemTc)) != cudaSuccess) return e;
    const size_t PN = (size_t)a.headdim * a.dstate;
    profile_kernel_begin(s);
    bwd_state_pass<<<dim3((unsigned)((PN + kThreads - 1) / kThreads), H, a.batch), kThreads, 0, s>>>(a);
    profile_kernel_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    int sms = 148;
    if ((e = sm_count(&sms)) != cudaSuccess) return e;
    const long long btiles = (long long)a.nchunks * H * a.batch;  // persistent: one CTA per SM
    profile_kernel_begin(s);
    tcb::bwd_chunk_tc<<<(unsigned)std::min<long long>(btiles, sms), tcb::kTc, tcb::kSmemTc, s>>>(xm, dym, bm, cm, dbm,
                                                                                             dcm, dxm, a);
    profile_kernel_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_reductions(a, s);
}

template <typename T>
cudaError_t launch_bwd_dtype(const BwdArgs &a, cudaStream_t s)
{
    if (a.headdim <= 16) return launch_bwd_typed<T, 1>(a, s);
    if (a.headdim <= 32) return launch_bwd_typed<T, 2>(a, s);
    if (a.headdim <= 64) return launch_bwd_typed<T, 4>(a, s);
    return launch_bwd_typed<T, 8>(a, s);
}

bool aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

// The tensor-core path: bf16, headdim 64, dstate 64, TMA-aligned inputs.
bool use_tc(const BwdProblem &p)
{
    return p.dtype == SSD_DTYPE_BF16 && p.headdim == 64 && p.dstate == 64 && aligned16(p.x) && aligned16(p.dy) &&
           aligned16(p.B) && aligned16(p.C);
}

int chunk_len(const BwdProblem &p) { return use_tc(p) ? tcb::kQ : kBQ; }

// On the tensor-core path, S_c comes from the forward's chunk-state kernel when
// its head pairs (128 TMEM lanes = 2 heads of 64) fall inside one group.
bool fwd_states(const BwdProblem &p) { return use_tc(p) && p.nheads % 2 == 0 && (p.nheads / p.ngroups) % 2 == 0; }

}  // namespace

size_t bwd_workspace_bytes(const BwdProblem &p)
{
    const int q = chunk_len(p);
    const size_t nc = (size_t)(p.seqlen + q - 1) / q;
    const size_t units = (size_t)p.batch * p.nheads * nc;
    size_t v = 2 * align256(units * p.headdim * p.dstate * sizeof(float)) + align256(units * sizeof(float)) +
               2 * align256((size_t)p.batch * nc * p.nheads * sizeof(float));
    if (p.nheads != p.ngroups)
        v += 2 * align256((size_t)p.batch * p.seqlen * p.nheads * p.dstate * sizeof(float));
    return v;
}

int bwd_kernel_count(const BwdProblem &p) { return (p.nheads != p.ngroups ? 5 : 4) + (fwd_states(p) ? 1 : 0); }

const char *bwd_kernel_names(const BwdProblem &p)
{
    if (fwd_states(p))
        return p.nheads != p.ngroups
                   ? "chunk_state_tc,chunk_state_tc,bwd_state_pass,bwd_chunk_tc,bwd_reduce_groups,bwd_reduce_heads"
                   : "chunk_state_tc,chunk_state_tc,bwd_state_pass,bwd_chunk_tc,bwd_reduce_heads";
    if (use_tc(p))
        return p.nheads != p.ngroups
                   ? "bwd_chunk_states,bwd_state_pass,bwd_chunk_tc,bwd_reduce_groups,bwd_reduce_heads"
                   : "bwd_chunk_states,bwd_state_pass,bwd_chunk_tc,bwd_reduce_heads";
    return p.nheads != p.ngroups ? "bwd_chunk_states,bwd_state_pass,bwd_chunk,bwd_reduce_groups,bwd_reduce_heads"
                                 : "bwd_chunk_states,bwd_state_pass,bwd_chunk,bwd_reduce_heads";
}

cudaError_t launch_bwd(const BwdProblem &p, void *workspace, cudaStream_t s)
{
    BwdArgs a;
    a.x = p.x;
    a.dt = p.dt;
    a.A = p.A;
    a.B = p.B;
    a.C = p.C;
    a.D = p.D;
    a.init_state = p.init_state;
    a.dy = p.dy;
    a.dfinal = p.dfinal;
    a.dx = p.dx;
    a.ddt = p.ddt;
    a.dA = p.dA;
    a.dB = p.dB;
    a.dC = p.dC;
    a.dD = p.dD;
    a.dinit = p.dinit;
    a.batch = p.batch;
    a.seqlen = p.seqlen;
    a.nheads = p.nheads;
    a.headdim = p.headdim;
    a.ngroups = p.ngroups;
    a.dstate = p.dstate;
    const int q = chunk_len(p);
    a.nchunks = (p.seqlen + q - 1) / q;
    a.err_word = p.err_word;
    const size_t units = (size_t)p.batch * p.nheads * a.nchunks;
    const size_t st = align256(units * p.headdim * p.dstate * sizeof(float));
    const size_t part = align256((size_t)p.batch * a.nchunks * p.nheads * sizeof(float));
    char *w = static_cast<char *>(workspace);
    a.hs = reinterpret_cast<float *>(w);
    a.gs = reinterpret_cast<float *>(w + st);
    a.decay = reinterpret_cast<float *>(w + 2 * st);
    a.dAp = reinterpret_cast<float *>(w + 2 * st + align256(units * sizeof(float)));
    a.dDp = reinterpret_cast<float *>(reinterpret_cast<char *>(a.dAp) + part);
    if (p.nheads != p.ngroups) {
        const size_t pp = align256((size_t)p.batch * p.seqlen * p.nheads * p.dstate * sizeof(float));
        a.dBp = reinterpret_cast<float *>(reinterpret_cast<char *>(a.dDp) + part);
        a.dCp = reinterpret_cast<float *>(reinterpret_cast<char *>(a.dBp) + pp);
    } else {
        a.dBp = a.dCp = nullptr;
    }
    if (use_tc(p)) return launch_bwd_tc(a, s);
    return p.dtype == SSD_DTYPE_BF16 ? launch_bwd_dtype<__nv_bfloat16>(a, s) : launch_bwd_dtype<float>(a, s);
}

}  // namespace ssd
