// ssd_step.cu -- one recurrent step of the SSD layer: the constant-size-state
// inference form ("深挖-Mamba", comparison table: no KV cache, only the fixed-size
// hidden state h_t is kept; section "Mamba-2 (2024)": training in the matrix
// form, inference in the recurrent form).
//
// For every (batch b, head h, headdim row p), with group g = h / (H / G):
//     a        = exp(dt[b,h] A[h])
//     h[n]     = a h[n] + dt[b,h] x[b,h,p] B[b,g,n]          (state, in place)
//     y[b,h,p] = sum_n C[b,g,n] h[n] + D[h] x[b,h,p]
// which is the recurrence of ssd_fwd for one token, the state being
// init_state on entry and final_state on exit.
//
// The step is bound by the state traffic (4 P N bytes read and written per
// (b, h)).  When dstate is a power of two from 4 to 128 and the state is
// 16-byte aligned, each thread owns 4 consecutive states of one row (16-byte
// loads and stores, streamed past L1) and the dstate/4 threads of a row reduce
// C . h with shuffles; otherwise one warp takes a row, lanes striding over n.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kStepV = 2;  // float4s of state per thread at large batch

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(256) ssd_step_kernel(const T *__restrict__ x, const float *__restrict__ dt,
                                                       const float *__restrict__ A, const T *__restrict__ B,
                                                       const T *__restrict__ C, const float *__restrict__ D,
                                                       float *__restrict__ state, T *__restrict__ y, int batch,
                                                       int H, int P, int G, int N)
{
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);  // (b, h, p)
    const long long rows = (long long)batch * H * P;
    if (row >= rows) return;
    const int h = (int)((row / P) % H);
    const int b = (int)(row / ((long long)P * H));
    const int g = h / (H / G);
    const float d = dt[(size_t)b * H + h];
    const float a = expf(d * A[h]);
    const float dx = d * to_f(x[row]);
    const T *Bg = B + ((size_t)b * G + g) * N;
    const T *Cg = C + ((size_t)b * G + g) * N;
    float *s = state + (size_t)row * N;
    float acc = 0.f;
    for (int n = lane; n < N; n += 32) {
        const float v = fmaf(a, s[n], dx * to_f(Bg[n]));
        s[n] = v;
        acc = fmaf(to_f(Cg[n]), v, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) y[row] = from_f<T>(acc + (D ? D[h] * to_f(x[row]) : 0.f));
}

// 4 states per thread; `lg` = log2(dstate / 4) threads per row (<= 5).
template <typename T>
__device__ __forceinline__ void load4(const T *p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float *p, float (&v)[4])
{
    const float4 t = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[4])
{
    const uint2 t = __ldg(reinterpret_cast<const uint2 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&t);
    const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    v[0] = a.x, v[1] = a.y, v[2] = b.x, v[3] = b.y;
}

// V float4s of one row per thread (4 V states), interleaved: thread q of the row
// owns float4s q, q + t, ..., t = 2^lg threads per row, dstate = 4 V t, so every
// load and store instruction of a warp is contiguous.  All V state loads are
// issued before any is used: each thread keeps 16 V bytes of the state stream
// in flight.
template <typename T, int V>
__global__ void __launch_bounds__(256) ssd_step_vec_kernel(const T *__restrict__ x, const float *__restrict__ dt,
                                                           const float *__restrict__ A, const T *__restrict__ B,
                                                           const T *__restrict__ C, const float *__restrict__ D,
                                                           float *__restrict__ state, T *__restrict__ y, int batch,
                                                           int H, int P, int G, int lg)
{
    // grid: (rows of one (b, h) x threads per row) / 256, H, batch -- no per-thread division
    const int h = blockIdx.y, b = blockIdx.z;
    const int lt = blockIdx.x * blockDim.x + threadIdx.x;  // thread within the (b, h) block of rows
    const int q = lt & ((1 << lg) - 1);                    // which 4 V states of the row
    const int p = lt >> lg;
    const bool live = p < P;
    const long long r = ((long long)b * H + h) * P + (live ? p : P - 1);  // dead threads still join the shuffles
    const int N = (4 * V) << lg;
    const int g = h / (H / G);
    const int tpr = 1 << lg;  // threads per row
    float4 *sp = reinterpret_cast<float4 *>(state + (size_t)r * N) + q;
    float4 sv[V];
#pragma unroll
    for (int k = 0; k < V; ++k) sv[k] = __ldcs(sp + k * tpr);
    const float d = __ldg(dt + (size_t)b * H + h);
    const float a = expf(d * __ldg(A + h));
    const float xv = to_f(x[r]);
    const float dx = d * xv;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
        float bv[4], cv[4];
        load4<T>(B + ((size_t)b * G + g) * N + 4 * (q + k * tpr), bv);
        load4<T>(C + ((size_t)b * G + g) * N + 4 * (q + k * tpr), cv);
        sv[k].x = fmaf(a, sv[k].x, dx * bv[0]);
        sv[k].y = fmaf(a, sv[k].y, dx * bv[1]);
        sv[k].z = fmaf(a, sv[k].z, dx * bv[2]);
        sv[k].w = fmaf(a, sv[k].w, dx * bv[3]);
        if (live) __stcs(sp + k * tpr, sv[k]);
        acc = fmaf(cv[0], sv[k].x, fmaf(cv[1], sv[k].y, fmaf(cv[2], sv[k].z, fmaf(cv[3], sv[k].w, acc))));
    }
    for (int o = 1; o < (1 << lg); o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (live && q == 0) y[r] = from_f<T>(acc + (D ? __ldg(D + h) * xv : 0.f));
}

template <typename T, int V>
void launch_vec(const void *x, const float *dt, const float *A, const void *B, const void *C, const float *D,
                float *state, void *y, int batch, int nheads, int headdim, int ngroups, int lg, cudaStream_t s)
{
    // the threads of one (b, h) -- headdim rows of 2^lg -- in blocks of at most 256, whole warps
    const int per = headdim << lg;
    const int block = per >= 256 ? 256 : (per + 31) / 32 * 32;
    const dim3 grid((unsigned)((per + block - 1) / block), (unsigned)nheads, (unsigned)batch);
    ssd_step_vec_kernel<T, V><<<grid, block, 0, s>>>(static_cast<const T *>(x), dt, A, static_cast<const T *>(B),
                                                   static_cast<const T *>(C), D, state, static_cast<T *>(y), batch,
                                                   nheads, headdim, ngroups, lg);
}

}  // namespace

cudaError_t launch_step(const void *x, const float *dt, const float *A, const void *B, const void *C,
                        const float *D, float *state, void *y, int batch, int nheads, int headdim, int ngroups,
                        int dstate, ssd_dtype_t dtype, cudaStream_t s)
{
    const long long rows = (long long)batch * nheads * headdim;
    // V float4s of state per thread: more bytes in flight per thread when there are
    // enough rows to fill the GPU anyway (one float4 per thread for small batches)
    const int V = (rows * dstate / 4 >= (1ll << 20) && dstate >= 4 * kStepV) ? kStepV : 1;
    int lg = -1;
    for (int k = 0; k <= 5; ++k)
        if (dstate == ((4 * V) << k)) lg = k;
    const bool al = (reinterpret_cast<uintptr_t>(state) & 15) == 0 && (reinterpret_cast<uintptr_t>(B) & 7) == 0 &&
                    (reinterpret_cast<uintptr_t>(C) & 7) == 0 &&
                    nheads <= 65535 && batch <= 65535 &&  // the vector kernel's grid is (.., nheads, batch)
                    ((long long)headdim << 5) < (1ll << 31);
    if (lg >= 0 && al && dtype == SSD_DTYPE_BF16) {
        if (V == 1)
            launch_vec<__nv_bfloat16, 1>(x, dt, A, B, C, D, state, y, batch, nheads, headdim, ngroups, lg, s);
        else
            launch_vec<__nv_bfloat16, kStepV>(x, dt, A, B, C, D, state, y, batch, nheads, headdim, ngroups, lg, s);
        return cudaGetLastError();
    }
    if (lg >= 0 && al && dtype == SSD_DTYPE_F32 && (reinterpret_cast<uintptr_t>(B) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(C) & 15) == 0) {
        if (V == 1)
            launch_vec<float, 1>(x, dt, A, B, C, D, state, y, batch, nheads, headdim, ngroups, lg, s);
        else
            launch_vec<float, kStepV>(x, dt, A, B, C, D, state, y, batch, nheads, headdim, ngroups, lg, s);
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)((rows + 7) / 8);  // 8 rows (warps) per block
    if (dtype == SSD_DTYPE_BF16)
        ssd_step_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(x), dt, A, static_cast<const __nv_bfloat16 *>(B),
            static_cast<const __nv_bfloat16 *>(C), D, state, static_cast<__nv_bfloat16 *>(y), batch, nheads,
            headdim, ngroups, dstate);
    else
        ssd_step_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(x), dt, A,
                                                    static_cast<const float *>(B), static_cast<const float *>(C), D,
                                                    state, static_cast<float *>(y), batch, nheads, headdim, ngroups,
                                                    dstate);
    return cudaGetLastError();
}

}  // namespace ssd
