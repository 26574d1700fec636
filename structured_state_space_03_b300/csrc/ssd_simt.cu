// ssd_simt.cu -- chunked SSD forward on fp32 FMA units (no tensor cores).
//
// This is the fp32 path (fp32 inputs need 1e-4 relative accuracy, which
// neither TF32 nor bf16 tensor cores give) and the general path for sizes the
// tensor-core kernels are not built for.  One CTA of 256 threads per
// (chunk, head, batch); the chunk algebra is written out in ssd_internal.cuh.
// The chunk-to-chunk state pass is here for both multi-kernel paths: state_pass
// writes fp32 entry states (this path), state_pass_hilo the bf16 hi + lo terms
// per 64-wide slice that the tcgen05 chunk-output kernel loads by TMA.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;       // token tile (rows i and columns j of the diagonal block)
constexpr int kStateOuts = 8;   // chunk-state outputs per thread per pass

// Segment sum of one chunk: cs[t] (in-chunk inclusive prefix of dt*A) and
// dt[t] into shared memory; returns cs of the chunk's last token.
__device__ __forceinline__ float chunk_segsum(const Problem &pr, int tb, int h, int t0, int len,
                                              float *cs_s, float *dt_s, float *warp_tot)
{
    const int tid = threadIdx.x;
    float dtv = 0.f;
    if (tid < len) dtv = __ldg(pr.dt + ((size_t)tb * pr.seqlen + t0 + tid) * pr.nheads + h);
    const float cs = block_inclusive_scan_256(dtv * __ldg(pr.A + h), warp_tot);
    if (tid < kMaxChunk) {
        cs_s[tid] = cs;
        dt_s[tid] = pr.dtin ? (tid < len ? __ldg(pr.dtin + ((size_t)tb * pr.seqlen + t0 + tid) * pr.nheads + h) : 0.f)
                            : dtv;  // input scale
    }
    __syncthreads();
    return cs_s[len - 1];
}

// S_c[p][n] = sum_j exp(cs_last - cs_j) dt_j x_j[p] B_j[n]; also exp(cs_last).
template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_state_simt(Problem pr, Workspace ws)
{
    extern __shared__ float smem[];
    __shared__ float warp_tot[8];
    const int h = blockIdx.y;
    const ChunkRef ref = chunk_ref(pr, blockIdx.x, blockIdx.z);
    const int L = pr.seqlen, H = pr.nheads, P = pr.headdim, N = pr.dstate, G = pr.ngroups;
    const int g = h / (H / G);
    const int b = ref.tb, t0 = ref.t0, len = ref.len;
    float *cs_s = smem;             // [256]
    float *dt_s = cs_s + kMaxChunk; // [256]
    float *w_s = dt_s + kMaxChunk;  // [256]
    float *x_s = w_s + kMaxChunk;   // [kTile][P], pre-scaled by w
    float *b_s = x_s + kTile * P;   // [kTile][N]
    const T *x = static_cast<const T *>(pr.x);
    const T *Bm = static_cast<const T *>(pr.B);
    const int tid = threadIdx.x;

    const float cs_last = chunk_segsum(pr, b, h, t0, len, cs_s, dt_s, warp_tot);
    if (tid < len) w_s[tid] = expf(cs_last - cs_s[tid]) * dt_s[tid];
    const size_t slot = state_slot(pr, ref, h);
    if (tid == 0) ws.decay[slot] = expf(cs_last);
    __syncthreads();

    const int PN = P * N;
    float *out = ws.states + slot * (size_t)PN;
    for (int o0 = 0; o0 < PN; o0 += kThreads * kStateOuts) {
        float acc[kStateOuts];
#pragma unroll
        for (int k = 0; k < kStateOuts; ++k) acc[k] = 0.f;
        for (int j0 = 0; j0 < len; j0 += kTile) {
            const int tj = min(kTile, len - j0);
            for (int e = tid; e < tj * P; e += kThreads) {
                const int jj = e / P, p = e - jj * P;
                x_s[e] = load_el(x, (((size_t)b * L + t0 + j0 + jj) * H + h) * P + p) * w_s[j0 + jj];
            }
            for (int e = tid; e < tj * N; e += kThreads) {
                const int jj = e / N, n = e - jj * N;
                b_s[e] = load_el(Bm, (((size_t)b * L + t0 + j0 + jj) * G + g) * N + n);
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kStateOuts; ++k) {
                const int o = o0 + tid + k * kThreads;
                if (o < PN) {
                    const int p = o / N, n = o - p * N;
                    float a = acc[k];
                    for (int jj = 0; jj < tj; ++jj) a = fmaf(x_s[jj * P + p], b_s[jj * N + n], a);
                    acc[k] = a;
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int k = 0; k < kStateOuts; ++k) {
            const int o = o0 + tid + k * kThreads;
            if (o < PN) out[o] = acc[k];
        }
    }
}

// y_i = sum_{j<=i} (C_i.B_j) exp(cs_i - cs_j) dt_j x_j + exp(cs_i) C_i.h_c + D x_i
template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_out_simt(Problem pr, Workspace ws)
{
    extern __shared__ float smem[];
    __shared__ float warp_tot[8];
    const int h = blockIdx.y;
    const ChunkRef ref = chunk_ref(pr, blockIdx.x, blockIdx.z);
    const int L = pr.seqlen, H = pr.nheads, P = pr.headdim, N = pr.dstate, G = pr.ngroups;
    const int g = h / (H / G);
    const int b = ref.tb, t0 = ref.t0, len = ref.len;
    float *cs_s = smem;                 // [256]
    float *dt_s = cs_s + kMaxChunk;     // [256]
    float *c_s = dt_s + kMaxChunk;      // [kTile][N]   C rows of the current i tile
    const int NB = N + 1;               // padded row stride of b_s (no bank conflicts)
    float *b_s = c_s + kTile * N;       // [kTile][NB]  B rows of the current j tile
    float *x_s = b_s + kTile * NB;      // [kTile][P]   x rows of the current j tile
    float *s_s = x_s + kTile * P;       // [kTile][kTile+1] masked, decayed C.B
    float *h_s = s_s + kTile * (kTile + 1);  // [P][kTile+1] slice of h_c over n
    const T *x = static_cast<const T *>(pr.x);
    const T *Bm = static_cast<const T *>(pr.B);
    const T *Cm = static_cast<const T *>(pr.C);
    T *y = static_cast<T *>(pr.y);
    const int tid = threadIdx.x;
    const float *hc = ws.states + state_slot(pr, ref, h) * (size_t)P * N;
    const float Dh = pr.D ? __ldg(pr.D + h) : 0.f;

    chunk_segsum(pr, b, h, t0, len, cs_s, dt_s, warp_tot);

    constexpr int kOuts = kTile * kMaxHeaddim / kThreads;  // 32
    for (int i0 = 0; i0 < len; i0 += kTile) {
        const int ti = min(kTile, len - i0);
        for (int e = tid; e < kTile * N; e += kThreads) {
            const int ii = e / N, n = e - ii * N;
            c_s[e] = ii < ti ? load_el(Cm, (((size_t)b * L + t0 + i0 + ii) * G + g) * N + n) : 0.f;
        }
        float acc[kOuts];
#pragma unroll
        for (int k = 0; k < kOuts; ++k) acc[k] = 0.f;

        // off-diagonal blocks: C_i . h_c, over n in slices of kTile
        for (int n0 = 0; n0 < N; n0 += kTile) {
            const int tn = min(kTile, N - n0);
            __syncthreads();
            for (int e = tid; e < P * kTile; e += kThreads) {
                const int p = e / kTile, nn = e - p * kTile;
                h_s[p * (kTile + 1) + nn] = nn < tn ? hc[(size_t)p * N + n0 + nn] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kOuts; ++k) {
                const int o = tid + k * kThreads;
                if (o < kTile * P) {
                    const int ii = o / P, p = o - ii * P;
                    float a = acc[k];
                    for (int nn = 0; nn < tn; ++nn) a = fmaf(c_s[ii * N + n0 + nn], h_s[p * (kTile + 1) + nn], a);
                    acc[k] = a;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kOuts; ++k) {
            const int o = tid + k * kThreads;
            if (o < kTile * P) {
                const int ii = o / P;
                acc[k] *= ii < ti ? expf(cs_s[i0 + ii]) : 0.f;
            }
        }

        // diagonal block: j tiles up to the end of this i tile
        for (int j0 = 0; j0 < i0 + ti; j0 += kTile) {
            const int tj = min(kTile, i0 + ti - j0);
            __syncthreads();
            for (int e = tid; e < kTile * N; e += kThreads) {
                const int jj = e / N, n = e - jj * N;
                b_s[jj * NB + n] = jj < tj ? load_el(Bm, (((size_t)b * L + t0 + j0 + jj) * G + g) * N + n) : 0.f;
            }
            for (int e = tid; e < kTile * P; e += kThreads) {
                const int jj = e / P, p = e - jj * P;
                x_s[e] = jj < tj ? load_el(x, (((size_t)b * L + t0 + j0 + jj) * H + h) * P + p) : 0.f;
            }
            __syncthreads();
            for (int e = tid; e < kTile * kTile; e += kThreads) {
                const int ii = e / kTile, jj = e - ii * kTile;
                const int i = i0 + ii, j = j0 + jj;
                float v = 0.f;
                if (ii < ti && jj < tj && j <= i) {
                    float d = 0.f;
                    for (int n = 0; n < N; ++n) d = fmaf(c_s[ii * N + n], b_s[jj * NB + n], d);
                    v = d * expf(cs_s[i] - cs_s[j]) * dt_s[j];
                }
                s_s[ii * (kTile + 1) + jj] = v;
            }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < kOuts; ++k) {
                const int o = tid + k * kThreads;
                if (o < kTile * P) {
                    const int ii = o / P, p = o - ii * P;
                    float a = acc[k];
                    for (int jj = 0; jj < tj; ++jj) a = fmaf(s_s[ii * (kTile + 1) + jj], x_s[jj * P + p], a);
                    acc[k] = a;
                }
            }
        }

        // skip term and store
#pragma unroll
        for (int k = 0; k < kOuts; ++k) {
            const int o = tid + k * kThreads;
            if (o < kTile * P) {
                const int ii = o / P, p = o - ii * P;
                if (ii < ti) {
                    const size_t idx = (((size_t)b * L + t0 + i0 + ii) * H + h) * P + p;
                    store_el(y, idx, acc[k] + Dh * load_el(x, idx));
                }
            }
        }
        __syncthreads();
    }
}

// h_c (state entering chunk c) for every chunk, in place over S_c; final state.
__global__ void __launch_bounds__(kThreads) state_pass(Problem pr, Workspace ws)
{
    const int PN = pr.headdim * pr.dstate;
    const int e = blockIdx.x * kThreads + threadIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    if (e >= PN) return;
    const size_t bh = (size_t)b * pr.nheads + h;
    float st = pr.init_state ? pr.init_state[bh * PN + e] : 0.f;
    // batch layout: the nchunks chunks of (b, h); packed: sequence b's chunks, a
    // contiguous range of the sequence-major numbering in the layout [1][H][total]
    const size_t first = pr.chunks ? (size_t)h * pr.total_chunks + pr.seq_first[b] : bh * pr.nchunks;
    float *s = ws.states + first * (size_t)PN + e;
    const float *dec = ws.decay + first;
    // Chunk states go in batches of kAhead, double-buffered: the next batch's loads
    // are issued before the current batch is applied and overwritten, so each thread
    // keeps kAhead independent loads in flight at all times (batches of 8 measured
    // best: 0.49 -> 0.29 ms on 512 chunks x 24 heads x 64 x 256)
    constexpr int kAhead = 8;
    const int nc = pr.chunks ? pr.seq_first[b + 1] - pr.seq_first[b] : pr.nchunks;
    float sc[kAhead], dk[kAhead];
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {
        if (k < nc) {
            sc[k] = s[(size_t)k * PN];
            dk[k] = __ldg(dec + k);
        }
    }
    for (int c0 = 0; c0 < nc; c0 += kAhead) {
        float sn[kAhead], dn[kAhead];
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            if (c0 + kAhead + k < nc) {
                sn[k] = s[(size_t)(c0 + kAhead + k) * PN];
                dn[k] = __ldg(dec + c0 + kAhead + k);
            }
        }
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            if (c0 + k < nc) {
                s[(size_t)(c0 + k) * PN] = st;
                st = fmaf(dk[k], st, sc[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            sc[k] = sn[k];
            dk[k] = dn[k];
        }
    }
    if (pr.final_state) pr.final_state[bh * PN + e] = st;
}

// The same pass for the tcgen05 chunk-output kernel, which takes h_c as two bf16
// terms (hi = bf16(h), lo = bf16(h - hi); a single rounding of a carried state can
// cost ~2% of RMS(y)).  They are written in place of the fp32 values, per 64-wide
// slice of the state dimension: row p of a slot, viewed as 2 NS bf16, holds for
// slice s the 64 hi values at [128 s, 128 s + 64) and the 64 lo values at
// [128 s + 64, 128 s + 128) -- the 256 bytes the slice's fp32 values occupied, so the
// chunk-output kernel loads both operands by TMA as they are.  A warp owns one
// (row, slice) block: lane l reads fp32 words l and l + 32 of it and carries elements
// 2l and 2l + 1 (their chunk states come from the lanes that read them, by shuffles),
// so every lane overwrites exactly the two words it read itself.
__global__ void __launch_bounds__(kThreads) state_pass_hilo(Problem pr, Workspace ws)
{
    const int PN = pr.headdim * pr.dstate;
    const int lane = threadIdx.x & 31;
    const int blk = (int)((blockIdx.x * kThreads + threadIdx.x) >> 5);  // 64-element block of the slot
    const int h = blockIdx.y, b = blockIdx.z;
    if (blk * 64 >= PN) return;  // warp-uniform
    const size_t bh = (size_t)b * pr.nheads + h;
    const int ea = blk * 64 + 2 * lane;  // the two elements this lane carries
    float st0 = pr.init_state ? pr.init_state[bh * PN + ea] : 0.f;
    float st1 = pr.init_state ? pr.init_state[bh * PN + ea + 1] : 0.f;
    const size_t first = pr.chunks ? (size_t)h * pr.total_chunks + pr.seq_first[b] : bh * pr.nchunks;
    float *s = ws.states + first * (size_t)PN + blk * 64;
    const float *dec = ws.decay + first;
    const int nc = pr.chunks ? pr.seq_first[b + 1] - pr.seq_first[b] : pr.nchunks;
    const int src0 = (2 * lane) & 31, src1 = (2 * lane + 1) & 31;
    const bool upper = lane >= 16;  // elements 2 lane, 2 lane + 1 lie in the block's second half
    // batches of kAhead chunks, double-buffered as in state_pass
    constexpr int kAhead = 8;
    float w0[kAhead], w1[kAhead], dk[kAhead];
#pragma unroll
    for (int k = 0; k < kAhead; ++k) {
        if (k < nc) {
            w0[k] = s[(size_t)k * PN + lane];
            w1[k] = s[(size_t)k * PN + 32 + lane];
            dk[k] = __ldg(dec + k);
        }
    }
    for (int c0 = 0; c0 < nc; c0 += kAhead) {
        float n0[kAhead], n1[kAhead], dn[kAhead];
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            if (c0 + kAhead + k < nc) {
                n0[k] = s[(size_t)(c0 + kAhead + k) * PN + lane];
                n1[k] = s[(size_t)(c0 + kAhead + k) * PN + 32 + lane];
                dn[k] = __ldg(dec + c0 + kAhead + k);
            }
        }
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            if (c0 + k < nc) {  // warp-uniform
                const float a0 = __shfl_sync(0xffffffffu, w0[k], src0), a1 = __shfl_sync(0xffffffffu, w1[k], src0);
                const float b0 = __shfl_sync(0xffffffffu, w0[k], src1), b1 = __shfl_sync(0xffffffffu, w1[k], src1);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(st0, st1);
                const float2 hf = __bfloat1622float2(hi);
                const __nv_bfloat162 lo = __floats2bfloat162_rn(st0 - hf.x, st1 - hf.y);
                uint32_t *slot = reinterpret_cast<uint32_t *>(s + (size_t)(c0 + k) * PN);
                slot[lane] = *reinterpret_cast<const uint32_t *>(&hi);
                slot[32 + lane] = *reinterpret_cast<const uint32_t *>(&lo);
                st0 = fmaf(dk[k], st0, upper ? a1 : a0);
                st1 = fmaf(dk[k], st1, upper ? b1 : b0);
            }
        }
#pragma unroll
        for (int k = 0; k < kAhead; ++k) {
            w0[k] = n0[k];
            w1[k] = n1[k];
            dk[k] = dn[k];
        }
    }
    if (pr.final_state) {
        pr.final_state[bh * PN + ea] = st0;
        pr.final_state[bh * PN + ea + 1] = st1;
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    return ensure_smem_limit(reinterpret_cast<const void *>(kernel), bytes);
}

}  // namespace

cudaError_t launch_chunk_state_simt(const Problem &pr, const Workspace &ws, cudaStream_t s)
{
    const size_t smem = sizeof(float) * (3 * kMaxChunk + kTile * (pr.headdim + pr.dstate));
    const dim3 grid(pr.chunks ? pr.total_chunks : pr.nchunks, pr.nheads, pr.chunks ? 1 : pr.batch);
    cudaError_t e;
    if (pr.dtype == SSD_DTYPE_F32) {
        if ((e = set_smem(chunk_state_simt<float>, smem)) != cudaSuccess) return e;
        profile_kernel_begin(s);
        chunk_state_simt<float><<<grid, kThreads, smem, s>>>(pr, ws);
        profile_kernel_end(s);
    } else {
        if ((e = set_smem(chunk_state_simt<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        profile_kernel_begin(s);
        chunk_state_simt<__nv_bfloat16><<<grid, kThreads, smem, s>>>(pr, ws);
        profile_kernel_end(s);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_out_simt(const Problem &pr, const Workspace &ws, cudaStream_t s)
{
    const size_t smem = sizeof(float) * (2 * kMaxChunk + kTile * (2 * pr.dstate + 1 + pr.headdim) +
                                         kTile * (kTile + 1) + pr.headdim * (kTile + 1));
    const dim3 grid(pr.chunks ? pr.total_chunks : pr.nchunks, pr.nheads, pr.chunks ? 1 : pr.batch);
    cudaError_t e;
    if (pr.dtype == SSD_DTYPE_F32) {
        if ((e = set_smem(chunk_out_simt<float>, smem)) != cudaSuccess) return e;
        profile_kernel_begin(s);
        chunk_out_simt<float><<<grid, kThreads, smem, s>>>(pr, ws);
        profile_kernel_end(s);
    } else {
        if ((e = set_smem(chunk_out_simt<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        profile_kernel_begin(s);
        chunk_out_simt<__nv_bfloat16><<<grid, kThreads, smem, s>>>(pr, ws);
        profile_kernel_end(s);
    }
    return cudaGetLastError();
}

cudaError_t launch_state_pass(const Problem &pr, const Workspace &ws, cudaStream_t s, bool hilo)
{
    const int PN = pr.headdim * pr.dstate;
    profile_kernel_begin(s);
    if (hilo) {  // one warp per 64-element block (PN is a multiple of 64 on the tcgen05 path)
        const dim3 grid((PN / 2 + kThreads - 1) / kThreads, pr.nheads, pr.batch);
        state_pass_hilo<<<grid, kThreads, 0, s>>>(pr, ws);
    } else {
        const dim3 grid((PN + kThreads - 1) / kThreads, pr.nheads, pr.batch);
        state_pass<<<grid, kThreads, 0, s>>>(pr, ws);
    }
    profile_kernel_end(s);
    return cudaGetLastError();
}

}  // namespace ssd
