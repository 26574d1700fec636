// ssd_pre.cu -- per-(token, head) pre-step of the scan's two scalar inputs.
//
// The layer's discretisation ("Mamba模型：线性复杂度序列建模的革命性突破" §2.2 and
// "Mamba 模型" §2.3.1: zero-order hold, Abar = exp(dt A),
// Bbar = (dt A)^-1 (exp(dt A) - 1) dt B; §3.2 of the first page: the step dt is
// produced through a softplus) reduces, for a scalar A per head, to two
// per-(b, t, h) scalars: the step dt_eff that sets the decay exp(dt_eff A), and
// the scale of the input x_t B_t,
//     dt_eff   = softplus(dt + bias[h])   (or dt + bias[h] without the softplus)
//     scale    = expm1(dt_eff A) / A      (zero-order hold; dt_eff when A = 0)
//              = dt_eff                   (the simplified input dt B)
// This kernel writes them once; the scan kernels then read dt_eff in place of
// dt and, for the zero-order hold, the scale wherever dt multiplies the input.
#include <algorithm>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

__global__ void __launch_bounds__(256) pre_kernel(const float *__restrict__ dt, const float *__restrict__ bias,
                                                  const float *__restrict__ A, int flags, float *__restrict__ dt_eff,
                                                  float *__restrict__ scale, long long n, int H)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int h = (int)(i % H);
        const float z = dt[i] + (bias ? bias[h] : 0.f);
        // softplus(z) = max(z, 0) + log(1 + exp(-|z|)), without overflow
        const float d = (flags & kPreSoftplus) ? fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))) : z;
        dt_eff[i] = d;
        if (flags & kPreZoh) {
            const float a = A[h];
            scale[i] = a != 0.f ? expm1f(d * a) / a : d;
        }
    }
}

}  // namespace

cudaError_t launch_pre(const float *dt, const float *dt_bias, const float *A, int flags, float *dt_eff,
                       float *scale, int batch, int seqlen, int nheads, cudaStream_t s)
{
    const long long n = (long long)batch * seqlen * nheads;
    const unsigned grid = (unsigned)std::min<long long>((n + 255) / 256, 148LL * 16);
    pre_kernel<<<grid, 256, 0, s>>>(dt, dt_bias, A, flags, dt_eff, scale, n, nheads);
    return cudaGetLastError();
}

}  // namespace ssd
