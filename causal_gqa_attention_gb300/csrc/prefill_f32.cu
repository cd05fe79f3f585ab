// prefill_f32.cu -- fused attention forward in fp32 on CUDA cores (fp32 inputs and output).
//
// The fp32 entry point promises results within about 1e-5 of exact arithmetic, which rules
// out the tensor cores' reduced-precision fp32 (tf32) path; every product, sum and
// exponential here is an fp32 FFMA/FADD/expf.
//
// Structure (one thread block = 64 query rows of one head; 4 threads per row, each holding a
// quarter of the head dims, interleaved so that shared-memory reads are conflict-free):
//   for each key tile of BN rows: stage K and V in shared memory, compute the BN scores of
//   each row (partial dot products summed over the 4 threads of the row), apply the causal
//   and length masks as -inf, then the online-softmax update m_new = max(m, tile max),
//   c = exp(m - m_new), l = l c + sum exp(s - m_new), acc = acc c + sum exp(s - m_new) v.
//   At the end O = acc / l and LSE = m + log l.
// Sources: "Attention three-op fusion" (xdnf.cn/news/349386) sections 2.2-2.3 (recurrence),
// 4.1-4.2 (K/V blocks staged in shared memory, output accumulator distributed over threads in
// registers, two block-wide synchronisations per tile), 4.3 (causal mask and fully masked
// tiles skipped), 6.1 (tail tile: out-of-range loads are 0 and their scores -inf).
#include "internal.h"

#include <cmath>

namespace gqa {
namespace {

constexpr int kRows = 64;         // query rows per block
constexpr int kThreads = kRows * 4;

template <int D, int BN>
__global__ void __launch_bounds__(kThreads)
    prefill_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                       const float *__restrict__ v, float *__restrict__ o, float *__restrict__ lse,
                       int S, int Hq, int Hkv, float scale, int causal)
{
    constexpr int DP = D / 4;  // dims per thread: part, part + 4, part + 8, ...
    __shared__ __align__(16) float Ks[BN][D];
    __shared__ __align__(16) float Vs[BN][D];

    const int nrb = (S + kRows - 1) / kRows;
    const int rb = causal ? (nrb - 1 - (int)blockIdx.x) : (int)blockIdx.x;  // long rows first
    const int h = blockIdx.y, b = blockIdx.z;
    const int g = h / (Hq / Hkv);
    const int r0 = rb * kRows;
    const int row = r0 + threadIdx.x / 4;
    const int part = threadIdx.x % 4;
    const bool live = row < S;

    const float *qrow = q + (((size_t)b * Hq + h) * S + (live ? row : 0)) * D;
    float qr[DP], acc[DP];
#pragma unroll
    for (int c = 0; c < DP; ++c) {
        qr[c] = live ? qrow[part + 4 * c] : 0.f;
        acc[c] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    const float *kh = k + ((size_t)b * Hkv + g) * (size_t)S * D;
    const float *vh = v + ((size_t)b * Hkv + g) * (size_t)S * D;
    const int last_key = causal ? min(S - 1, r0 + kRows - 1) : S - 1;
    const int ntiles = last_key / BN + 1;

    for (int t = 0; t < ntiles; ++t) {
        const int k0 = t * BN;
        __syncthreads();  // previous tile fully consumed
        for (int idx = threadIdx.x; idx < BN * D / 4; idx += kThreads) {
            const int jj = idx / (D / 4), c4 = idx % (D / 4);
            float4 kv4 = make_float4(0.f, 0.f, 0.f, 0.f), vv4 = kv4;
            if (k0 + jj < S) {
                kv4 = reinterpret_cast<const float4 *>(kh + (size_t)(k0 + jj) * D)[c4];
                vv4 = reinterpret_cast<const float4 *>(vh + (size_t)(k0 + jj) * D)[c4];
            }
            reinterpret_cast<float4 *>(&Ks[jj][0])[c4] = kv4;
            reinterpret_cast<float4 *>(&Vs[jj][0])[c4] = vv4;
        }
        __syncthreads();  // tile staged

        float s[BN];
#pragma unroll
        for (int jj = 0; jj < BN; ++jj) {
            float d = 0.f;
#pragma unroll
            for (int c = 0; c < DP; ++c) d = fmaf(qr[c], Ks[jj][part + 4 * c], d);
            d += __shfl_xor_sync(0xffffffffu, d, 1);
            d += __shfl_xor_sync(0xffffffffu, d, 2);
            const int key = k0 + jj;
            s[jj] = (key >= S || (causal && key > row)) ? -INFINITY : d * scale;
        }
        float tmax = s[0];
#pragma unroll
        for (int jj = 1; jj < BN; ++jj) tmax = fmaxf(tmax, s[jj]);
        const float mn = fmaxf(m, tmax);
        const float mu = (mn == -INFINITY) ? 0.f : mn;
        const float corr = expf(m - mu);
        l *= corr;
#pragma unroll
        for (int c = 0; c < DP; ++c) acc[c] *= corr;
#pragma unroll
        for (int jj = 0; jj < BN; ++jj) {
            const float p = expf(s[jj] - mu);
            l += p;
#pragma unroll
            for (int c = 0; c < DP; ++c) acc[c] = fmaf(p, Vs[jj][part + 4 * c], acc[c]);
        }
        m = mn;
    }

    if (live) {
        float *orow = o + (((size_t)b * Hq + h) * S + row) * D;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c = 0; c < DP; ++c) orow[part + 4 * c] = acc[c] * inv;
        if (lse != nullptr && part == 0)
            lse[((size_t)b * Hq + h) * S + row] = l > 0.f ? m + logf(l) : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, float *o,
                               float *lse, int B, int S, int Hq, int Hkv, int D, float scale,
                               int causal, cudaStream_t st)
{
    dim3 grid((S + kRows - 1) / kRows, Hq, B);
    if (D == 64)
        prefill_f32_kernel<64, 64><<<grid, kThreads, 0, st>>>(q, k, v, o, lse, S, Hq, Hkv, scale,
                                                              causal);
    else
        prefill_f32_kernel<128, 32><<<grid, kThreads, 0, st>>>(q, k, v, o, lse, S, Hq, Hkv,
                                                               scale, causal);
    return cudaGetLastError();
}

}  // namespace gqa
