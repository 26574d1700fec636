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
// Kernels (all fp32 FMA; one CTA of 256 threads per (chunk, head, batch)):
//   1. bwd_chunk_states  S_c, G_c and the chunk decays
//   2. bwd_state_pass    h_c forward and g_c backward over the chunks, dinit
//   3. bwd_chunk         the in-chunk terms above, dx, ddt, per-head dB / dC,
//                        per-chunk dA / dD parts
//   4. bwd_reduce        dB / dC over the heads of a group (when a group has
//                        more than one head), dA / dD over batch and chunks
// Every reduction runs in a fixed order, so results are bitwise reproducible.
#include <algorithm>

#include "ssd_internal.cuh"

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
};

// In-chunk prefix sums of dt*A (cs) and dt (cum) for the kBQ tokens from t0.
__device__ __forceinline__ void chunk_scalars(const BwdArgs &a, int b, int h, int t0, int len, float *cs_s,
                                              float *dt_s, float *cum_s, float *warp_tot)
{
    const int tid = threadIdx.x;
    float dtv = 0.f;
    if (tid < len) dtv = __ldg(a.dt + ((size_t)b * a.seqlen + t0 + tid) * a.nheads + h);
    const float cs = block_inclusive_scan_256(dtv * __ldg(a.A + h), warp_tot);
    const float cum = block_inclusive_scan_256(dtv, warp_tot);
    if (tid < kBQ) {
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
template <typename T, int MP>
__global__ void __launch_bounds__(kThreads) bwd_chunk_states(BwdArgs a)
{
    extern __shared__ float sm[];
    __shared__ float warp_tot[8];
    __shared__ float cs_s[kBQ], dt_s[kBQ], cum_s[kBQ];
    constexpr int PP = MP * 16;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int L = a.seqlen, H = a.nheads, P = a.headdim, N = a.dstate, G = a.ngroups;
    const int g = h / (H / G);
    const int t0 = c * kBQ, len = min(kBQ, L - t0);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float *xs = sm;               // [kBQ][PP]  x_j e^{cs_end - cs_j} dt_j
    float *ys = xs + kBQ * PP;    // [kBQ][PP]  dy_i e^{cs_i}
    float *bs = ys + kBQ * PP;    // [kBQ][kNT]
    float *cm = bs + kBQ * kNT;   // [kBQ][kNT]
    const T *x = static_cast<const T *>(a.x);
    const T *dy = static_cast<const T *>(a.dy);
    const T *Bm = static_cast<const T *>(a.B);
    const T *Cm = static_cast<const T *>(a.C);

    chunk_scalars(a, b, h, t0, len, cs_s, dt_s, cum_s, warp_tot);
    const float cs_end = cs_s[len - 1];
    const size_t bh = (size_t)b * H + h;
    if (tid == 0) a.decay[bh * a.nchunks + c] = expf(cs_end);
    for (int e = tid; e < kBQ * PP; e += kThreads) {
        const int t = e / PP, p = e - t * PP;
        float xv = 0.f, yv = 0.f;
        if (t < len && p < P) {
            const size_t i = (((size_t)b * L + t0 + t) * H + h) * P + p;
            xv = load_el(x, i) * (expf(cs_end - cs_s[t]) * dt_s[t]);
            yv = load_el(dy, i) * expf(cs_s[t]);
        }
        xs[e] = xv;
        ys[e] = yv;
    }
    float *S = a.hs + (bh * a.nchunks + c) * (size_t)P * N;
    float *Gc = a.gs + (bh * a.nchunks + c) * (size_t)P * N;
    for (int n0 = 0; n0 < N; n0 += kNT) {
        __syncthreads();  // xs / ys written; the previous pass's readers of bs / cm done
        for (int e = tid; e < kBQ * kNT; e += kThreads) {
            const int t = e / kNT, n = n0 + (e - t * kNT);
            float bv = 0.f, cv = 0.f;
            if (t < len && n < N) {
                const size_t i = (((size_t)b * L + t0 + t) * G + g) * N + n;
                bv = load_el(Bm, i);
                cv = load_el(Cm, i);
            }
            bs[e] = bv;
            cm[e] = cv;
        }
        __syncthreads();
        float accS[MP][4], accG[MP][4];
#pragma unroll
        for (int i = 0; i < MP; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) accS[i][q] = accG[i][q] = 0.f;
        for (int t = 0; t < len; ++t) {
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
    float s = a.init_state ? a.init_state[bh * PN + e] : 0.f;
    float nxt = hs[0];
    for (int c = 0; c < nc; ++c) {
        const float cur = nxt;
        if (c + 1 < nc) nxt = hs[(size_t)(c + 1) * PN];
        hs[(size_t)c * PN] = s;
        s = fmaf(dec[c], s, cur);
    }
    float gv = a.dfinal ? a.dfinal[bh * PN + e] : 0.f;
    nxt = gs[(size_t)(nc - 1) * PN];
    for (int c = nc - 1; c >= 0; --c) {
        const float cur = nxt;
        if (c > 0) nxt = gs[(size_t)(c - 1) * PN];
        gs[(size_t)c * PN] = gv;
        gv = fmaf(dec[c], gv, cur);
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

    chunk_scalars(a, b, h, t0, len, cs_s, dt_s, cum_s, warp_tot);
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
// 4a. dB / dC: sum of the per-head parts over the heads of each group.
__global__ void __launch_bounds__(kThreads) bwd_reduce_groups(BwdArgs a)
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

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

template <int MP>
size_t chunk_states_smem() { return sizeof(float) * (2 * kBQ * MP * 16 + 2 * kBQ * kNT); }
template <int MP>
size_t chunk_smem() { return sizeof(float) * (2 * kBQ * (MP * 16 + 1) + 2 * kBQ * (kBQ + 1) + 2 * kBQ * (kNS + 1) + 2 * MP * 16 * (kNS + 1)); }

template <typename T, int MP>
cudaError_t launch_bwd_typed(const BwdArgs &a, cudaStream_t s)
{
    const dim3 grid(a.nchunks, a.nheads, a.batch);
    cudaError_t e;
    const size_t s1 = chunk_states_smem<MP>(), s3 = chunk_smem<MP>();
    if ((e = ensure_smem_limit((const void *)bwd_chunk_states<T, MP>, s1)) != cudaSuccess) return e;
    if ((e = ensure_smem_limit((const void *)bwd_chunk<T, MP>, s3)) != cudaSuccess) return e;
    profile_kernel_begin(s);
    bwd_chunk_states<T, MP><<<grid, kThreads, s1, s>>>(a);
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
    if (a.dBp) {
        int sms = 148;
        if ((e = sm_count(&sms)) != cudaSuccess) return e;
        const size_t total = (size_t)a.batch * a.seqlen * a.ngroups * a.dstate;
        const size_t want = (total + kThreads - 1) / kThreads;
        const unsigned blocks = (unsigned)std::min<size_t>(want, (size_t)sms * 8);
        profile_kernel_begin(s);
        bwd_reduce_groups<<<blocks, kThreads, 0, s>>>(a);
        profile_kernel_end(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    profile_kernel_begin(s);
    bwd_reduce_heads<<<a.nheads, kThreads, 0, s>>>(a);
    profile_kernel_end(s);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_bwd_dtype(const BwdArgs &a, cudaStream_t s)
{
    if (a.headdim <= 16) return launch_bwd_typed<T, 1>(a, s);
    if (a.headdim <= 32) return launch_bwd_typed<T, 2>(a, s);
    if (a.headdim <= 64) return launch_bwd_typed<T, 4>(a, s);
    return launch_bwd_typed<T, 8>(a, s);
}

}  // namespace

size_t bwd_workspace_bytes(const BwdProblem &p)
{
    const size_t nc = (size_t)(p.seqlen + kBQ - 1) / kBQ;
    const size_t units = (size_t)p.batch * p.nheads * nc;
    size_t v = 2 * align256(units * p.headdim * p.dstate * sizeof(float)) + align256(units * sizeof(float)) +
               2 * align256((size_t)p.batch * nc * p.nheads * sizeof(float));
    if (p.nheads != p.ngroups)
        v += 2 * align256((size_t)p.batch * p.seqlen * p.nheads * p.dstate * sizeof(float));
    return v;
}

int bwd_kernel_count(const BwdProblem &p) { return p.nheads != p.ngroups ? 5 : 4; }

const char *bwd_kernel_names(const BwdProblem &p)
{
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
    a.nchunks = (p.seqlen + kBQ - 1) / kBQ;
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
    return p.dtype == SSD_DTYPE_BF16 ? launch_bwd_dtype<__nv_bfloat16>(a, s) : launch_bwd_dtype<float>(a, s);
}

}  // namespace ssd
