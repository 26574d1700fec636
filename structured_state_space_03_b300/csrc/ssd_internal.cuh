// ssd_internal.cuh -- shared declarations of the CUDA side of libssd.
//
// Chunked evaluation of the SSD layer ("Mamba 模型" §4.1, block decomposition
// of the semiseparable matrix; "Mamba-2架构深度解析" §2.2, chunked hybrid mode).
// With Q = chunk, token t in chunk c = t / Q, and the in-chunk inclusive
// prefix sum of the log-decays
//
//     cs_t = sum_{k = cQ .. t} dt_k * A_h                    (segment sum)
//
// the recurrence h_t = exp(dt_t A) h_{t-1} + dt_t x_t B_t^T unrolls into
//
//     S_c     = sum_{j in c} exp(cs_last - cs_j) dt_j x_j B_j^T     chunk state
//     h_{c+1} = exp(cs_last) h_c + S_c,  h_0 = init_state           state passing
//     y_i     = sum_{j in c, j <= i} (C_i . B_j) exp(cs_i - cs_j) dt_j x_j   diagonal block
//             + exp(cs_i) C_i . h_c                                 off-diagonal blocks
//             + D_h x_i                                             skip
//
// where h_c is the state entering chunk c.  All exponents are differences of
// in-chunk prefix sums with the later index first, so they are <= 0 for A <= 0
// and never overflow.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// Device error word flags (OR-ed together; read and cleared by the host).
enum : unsigned int {
    kDevErrTimeout = 1u,  // a bounded wait gave up
    kDevErrBounds = 2u,   // a kernel-side consistency check failed
};

// One chunk of a packed variable-length sequence: sequence b, chunk c of it,
// its index in the sequence-major numbering of all chunks, its first token in
// the packed token dimension, its length, and whether it is the sequence's last.
struct ChunkDesc {
    int b, c, gchunk, tok0, len, last, pad0, pad1;
};

struct Problem {
    const void *x;
    const float *dt;          // step of each token: the decay is exp(dt A)
    const float *dtin;        // input scale of each token (same layout as dt); null: dt itself
    const float *A;
    const void *B;
    const void *C;
    const float *D;           // may be null
    const float *init_state;  // may be null
    void *y;
    float *final_state;       // may be null
    int batch, seqlen, nheads, headdim, ngroups, dstate, chunk;
    int nchunks;
    ssd_dtype_t dtype;
    // Packed variable-length sequences (null: the batch layout).  Then batch is
    // the number of sequences, seqlen the packed token count, every tensor's
    // token dimension is the packed one (batch dimension 1), and chunks[k],
    // k < total_chunks, lists the chunks in chunk-major order (every sequence's
    // chunk 0, then every chunk 1, ...).
    const ChunkDesc *chunks;
    int total_chunks;
    // Packed layout on the multi-kernel paths: seq_first[q] is the index, in the
    // sequence-major numbering of all chunks (ChunkDesc::gchunk), of sequence q's
    // first chunk; seq_first[batch] = total_chunks (device memory).
    const int *seq_first;
    unsigned int *err_word;   // device address of the error word
    // Failure-detection test settings (ssd_test_set_fault): the limit of every
    // bounded wait of the fused kernels, and the unit (index in the fused
    // workspace) whose look-back publications are withheld (-1: none).
    unsigned long long wait_ns;
    long long withhold;
    // chunk_state_tc only: 1 computes the backward's adjoint chunk states
    // G_c = sum_j exp(cs_j) x_j B_j^T (x, B given as dy, C) and leaves the decays alone.
    int adjoint_states;
};

// Workspace carved out of one device buffer.
struct Workspace {
    float *states;  // [batch][nheads][nchunks][headdim][dstate]: S_c, then h_c in place (fp32, or
                    // bf16 hi / lo per 64-wide slice on the tcgen05 path: launch_state_pass)
    float *decay;   // [batch][nheads][nchunks]: exp(cs_last) of each chunk
    uint32_t *ticket = nullptr;  // tile ticket of the persistent chunk_out_tc (zeroed per launch)
};
// (The packed layout uses [1][nheads][total_chunks] in the sequence-major chunk
// numbering instead of [batch][nheads][nchunks].)

// The chunk a CTA of the multi-kernel paths works on.  Batch layout: chunk cx
// of batch element bz.  Packed layout: entry cx of the chunk table (bz is 0).
struct ChunkRef {
    int seq;  // batch element or packed sequence
    int tb;   // batch coordinate of the token tensors (0 when packed)
    int t0;   // first token of the chunk within its batch row
    int len;  // tokens in the chunk
    int sb;   // batch coordinate of the chunk's state and decay (0 when packed)
    int sc;   // chunk coordinate of the chunk's state and decay
    int nct;  // chunk extent of the state layout
};

__device__ __forceinline__ ChunkRef chunk_ref(const Problem &pr, int cx, int bz)
{
    ChunkRef r;
    if (pr.chunks) {
        const ChunkDesc d = pr.chunks[cx];
        r.seq = d.b;
        r.tb = 0;
        r.t0 = d.tok0;
        r.len = d.len;
        r.sb = 0;
        r.sc = d.gchunk;
        r.nct = pr.total_chunks;
    } else {
        r.seq = bz;
        r.tb = bz;
        r.t0 = cx * pr.chunk;
        r.len = min(pr.chunk, pr.seqlen - r.t0);
        r.sb = bz;
        r.sc = cx;
        r.nct = pr.nchunks;
    }
    return r;
}

// Index of head h's state / decay of the chunk in the workspace (in states of
// headdim x dstate, or in floats of the decay array).
__device__ __forceinline__ size_t state_slot(const Problem &pr, const ChunkRef &r, int h)
{
    return ((size_t)r.sb * pr.nheads + h) * r.nct + r.sc;
}

size_t workspace_bytes(const Problem &pr);
Workspace carve_workspace(const Problem &pr, void *base);

// SIMT (fp32 FMA) chunked kernels: any dtype, headdim/dstate/chunk <= 256.
cudaError_t launch_chunk_state_simt(const Problem &pr, const Workspace &ws, cudaStream_t s);
cudaError_t launch_chunk_out_simt(const Problem &pr, const Workspace &ws, cudaStream_t s);
// tcgen05 tensor-core chunked kernels: bf16, headdim 64/128, dstate 64/128/256, chunk <= 256.
bool tc_supported(const Problem &pr);
cudaError_t launch_chunk_state_tc(const Problem &pr, const Workspace &ws, cudaStream_t s);
cudaError_t launch_chunk_out_tc(const Problem &pr, const Workspace &ws, cudaStream_t s);
// Single fused tcgen05 kernel with a decoupled look-back over published chunk
// states: bf16, headdim 64/128, dstate 64/128, chunk <= 128.
bool fused_supported(const Problem &pr);
size_t fused_workspace_bytes(const Problem &pr);
cudaError_t launch_fused_tc(const Problem &pr, void *workspace, cudaStream_t s);
// Sequence-pipelined fused kernel (ssd_seq.cu): dstate 64, the batch layout of
// the fused kernels; every CTA carries the recurrence of its own run of chunks
// on chip and exchanges states only where a sequence continues on the next CTA.
bool seq_supported(const Problem &pr);
size_t seq_workspace_bytes(const Problem &pr);
cudaError_t launch_seq_tc(const Problem &pr, void *workspace, cudaStream_t s);
// Sequential inter-chunk state passing, shared by the multi-kernel paths.
// hilo: write each entry state h_c in place as bf16 hi and lo terms per 64-wide slice
// of the state dimension (the layout chunk_out_tc loads); else as fp32
cudaError_t launch_state_pass(const Problem &pr, const Workspace &ws, cudaStream_t s, bool hilo);

// Backward (ssd_bwd.cu): gradients of a scalar loss given dL/dy and dL/d(final
// state); fp32 FMA kernels, headdim <= kBwdMaxHeaddim, dstate <= kMaxDstate.
struct BwdProblem {
    const void *x;
    const float *dt;
    const float *A;
    const void *B;
    const void *C;
    const float *D;           // may be null
    const float *init_state;  // may be null
    const void *dy;           // [batch][seqlen][nheads][headdim], element type dtype
    const float *dfinal;      // may be null
    float *dx, *ddt, *dA, *dB, *dC;
    float *dD;                // may be null
    float *dinit;             // may be null
    int batch, seqlen, nheads, headdim, ngroups, dstate;
    ssd_dtype_t dtype;
    unsigned int *err_word;   // device error word (a failed bounded wait sets kDevErrTimeout)
};
constexpr int kBwdMaxHeaddim = 128;
size_t bwd_workspace_bytes(const BwdProblem &p);
int bwd_kernel_count(const BwdProblem &p);
const char *bwd_kernel_names(const BwdProblem &p);
cudaError_t launch_bwd(const BwdProblem &p, void *workspace, cudaStream_t s);

// Host-side caches and the per-kernel timing hook (ssd_host.cu).
// A 3-D [batch][rows][width] tensor map (bf16 or fp32), box box_cols x box_rows x 1,
// 128-byte swizzle or none; identical requests reuse one encoded map.
cudaError_t cached_tensor_map(CUtensorMap *out, const void *ptr, bool bf16, int width, int rows, int batch,
                              int box_cols, int box_rows, bool swizzle128);
// Raise a kernel's dynamic shared-memory limit once per (device, kernel, size).
cudaError_t ensure_smem_limit(const void *func, size_t bytes);
// SM count of the current device (queried once).
cudaError_t sm_count(int *n);
constexpr int kMaxProfileEvents = 16;
void profile_set(void *const *events, int count);
void profile_forward_begin();               // at the start of every forward
void profile_kernel_begin(cudaStream_t s);  // right before a kernel launch, after its host setup
void profile_kernel_end(cudaStream_t s);    // right after it

constexpr int kMaxChunk = 256;
constexpr int kFusedTile = 128;  // tokens per tile (TMEM lanes) of the fused kernels
constexpr int kMaxHeaddim = 256;
constexpr int kMaxDstate = 256;

__device__ __forceinline__ float load_el(const float *p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float load_el(const __nv_bfloat16 *p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void store_el(float *p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_el(__nv_bfloat16 *p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// Inclusive prefix sum over a 256-thread block (warp shuffles, then the warp
// totals).  `warp_tot` is 8 floats of shared memory.  Every thread calls it.
__device__ __forceinline__ float block_inclusive_scan_256(float v, float *warp_tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float w = lane < 8 ? warp_tot[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        if (lane < 8) warp_tot[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += warp_tot[warp - 1];
    __syncthreads();  // warp_tot may be reused by the caller
    return v;
}

// Pre-step (ssd_pre.cu): dt_eff = softplus(dt + bias) (or dt + bias) and, for
// the zero-order-hold input, the scale expm1(dt_eff A) / A, per (b, t, h).
enum : int { kPreSoftplus = 1, kPreZoh = 2 };
cudaError_t launch_pre(const float *dt, const float *dt_bias, const float *A, int flags, float *dt_eff,
                       float *scale, int batch, int seqlen, int nheads, cudaStream_t s);

// One recurrent step (ssd_step.cu): state [batch][nheads][headdim][dstate] fp32 in place.
cudaError_t launch_step(const void *x, const float *dt, const float *A, const void *B, const void *C,
                        const float *D, float *state, void *y, int batch, int nheads, int headdim, int ngroups,
                        int dstate, ssd_dtype_t dtype, cudaStream_t s);

}  // namespace ssd
