// decode.cu -- single-token attention against a bf16 KV cache, split over key chunks.
//
// Stage 1 (decode_split_kernel): one thread block per (key chunk, kv head, query-head
// subgroup, sequence). Every K and V row of the chunk is read once from device memory with
// 16-byte loads and used by all query heads of the group, which is what makes grouped-query
// decode cheap: the cache traffic is per kv head, not per query head. The block keeps an
// online-softmax state (running max m, running sum l, unnormalised output) per query head
// and writes it to the workspace.
// Stage 2 (decode_merge_kernel): per (sequence, query head), the chunk states are combined
// with weights 2^(m_s - M), M = max m_s, in a fixed order (deterministic).
//
// Sources: "Attention three-op fusion" (xdnf.cn/news/349386) section 2.2 (running max and sum,
// correction factor, order-free merge), section 4.4 (keys split across thread blocks with a
// cross-block merge of the partial results); "Hand-written Triton decoder"
// (m.nlpx.cn/news/28229) section 2.1 (2 KV heads serve 8 query heads) and section 3.3 (partials
// in a separate buffer, reduced by a second small kernel instead of atomics).
#include "internal.h"
#include "ptx.cuh"

#include <cmath>

namespace gqa {
namespace {

constexpr int kSplitThreads = 128;
constexpr int kSplitWarps = kSplitThreads / 32;

// D: head dim; HG: query heads per block (divides Hq/Hkv); U: key rows per lane group per step.
template <int D, int HG, int U>
__global__ void __launch_bounds__(kSplitThreads)
    decode_split_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kc,
                        const __nv_bfloat16 *__restrict__ vc, const int *__restrict__ seqlens,
                        float *__restrict__ ws_o, float2 *__restrict__ ws_ml, int Hq, int Hkv,
                        int max_len, int chunk, int nsplit, float scale_log2,
                        unsigned *__restrict__ status)
{
    constexpr int LPK = D / 8;                  // lanes per key row, 8 dims (16 bytes) each
    constexpr int KPW = 32 / LPK;               // key rows per warp per step
    constexpr int KPB = KPW * kSplitWarps;      // key rows per block per step
    __shared__ float s_m[KPB][HG], s_l[KPB][HG];
    __shared__ __align__(16) float s_acc[KPB][HG][D];

    const int split = blockIdx.x;
    const int subgroups = gridDim.y / Hkv;      // (Hq / Hkv) / HG
    const int g = blockIdx.y / subgroups;
    const int h0 = g * (Hq / Hkv) + (blockIdx.y % subgroups) * HG;
    const int b = blockIdx.z;

    int L = seqlens[b];
    if (L < 0 || L > max_len) {
        if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) atomicOr(status, 1u);
        L = L < 0 ? 0 : max_len;
    }
    const int start = split * chunk;
    if (start >= L) return;  // uniform over the block
    const int end = min(start + chunk, L);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub = lane % LPK;                       // which 8 dims
    const int slot = warp * KPW + lane / LPK;         // which key row of each step

    // query fragments for the HG heads, pre-scaled so that scores come out in log2 units
    float qf[HG][8];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        const uint4 w = *reinterpret_cast<const uint4 *>(q + ((size_t)b * Hq + h0 + h) * D + sub * 8);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qf[h][2 * e] = bf16lo(ws[e]) * scale_log2;
            qf[h][2 * e + 1] = bf16hi(ws[e]) * scale_log2;
        }
    }

    float m[HG], l[HG], acc[HG][8];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;
    }

    const size_t head_off = ((size_t)b * Hkv + g) * (size_t)max_len * D + sub * 8;
    const __nv_bfloat16 *kb = kc + head_off;
    const __nv_bfloat16 *vb = vc + head_off;

    for (int jb = start; jb < end; jb += KPB * U) {  // trip count uniform over the block
        uint4 kw[U], vw[U];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = jb + u * KPB + slot;
            ok[u] = j < end;
            if (ok[u]) {
                kw[u] = ld_nc_na_v4(kb + (size_t)j * D);
                vw[u] = ld_nc_na_v4(vb + (size_t)j * D);
            } else {
                kw[u] = make_uint4(0, 0, 0, 0);
                vw[u] = make_uint4(0, 0, 0, 0);
            }
        }
        float s[U][HG];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t w4[4] = {kw[u].x, kw[u].y, kw[u].z, kw[u].w};
            float kf[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kf[2 * e] = bf16lo(w4[e]);
                kf[2 * e + 1] = bf16hi(w4[e]);
            }
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) d = fmaf(qf[h][e], kf[e], d);
                s[u][h] = d;
            }
        }
        // sum the partial dots over the LPK lanes of each key row
#pragma unroll
        for (int off = LPK / 2; off >= 1; off >>= 1)
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int h = 0; h < HG; ++h) s[u][h] += __shfl_xor_sync(0xffffffffu, s[u][h], off);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (!ok[u])
#pragma unroll
                for (int h = 0; h < HG; ++h) s[u][h] = -INFINITY;

        float vf[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t w4[4] = {vw[u].x, vw[u].y, vw[u].z, vw[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                vf[u][2 * e] = bf16lo(w4[e]);
                vf[u][2 * e + 1] = bf16hi(w4[e]);
            }
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) {
            float bm = s[0][h];
#pragma unroll
            for (int u = 1; u < U; ++u) bm = fmaxf(bm, s[u][h]);
            const float mn = fmaxf(m[h], bm);
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            const float alpha = ex2(m[h] - mu);
            l[h] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[h][e] *= alpha;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float p = ex2(s[u][h] - mu);
                l[h] += p;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(p, vf[u][e], acc[h][e]);
            }
            m[h] = mn;
        }
    }

    // combine the KPB key-slot states of this block
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        if (sub == 0) {
            s_m[slot][h] = m[h];
            s_l[slot][h] = l[h];
        }
        float4 *dst = reinterpret_cast<float4 *>(&s_acc[slot][h][sub * 8]);
        dst[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
        dst[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < HG * D; idx += kSplitThreads) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll 4
        for (int s2 = 0; s2 < KPB; ++s2) M = fmaxf(M, s_m[s2][h]);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f, a = 0.f;
#pragma unroll 4
        for (int s2 = 0; s2 < KPB; ++s2) {
            const float w = ex2(s_m[s2][h] - Mu);
            Ls = fmaf(w, s_l[s2][h], Ls);
            a = fmaf(w, s_acc[s2][h][d], a);
        }
        const size_t row = ((size_t)b * Hq + h0 + h) * nsplit + split;
        ws_o[row * D + d] = a;
        if (d == 0) ws_ml[row] = make_float2(M, Ls);
    }
}

template <bool OUT_F32>
__global__ void __launch_bounds__(128)
    decode_merge_kernel(const float *__restrict__ ws_o, const float2 *__restrict__ ws_ml,
                        const int *__restrict__ seqlens, void *__restrict__ o,
                        float *__restrict__ lse, int Hq, int D, int max_len, int chunk, int nsplit)
{
    const int bh = blockIdx.x;
    const int b = bh / Hq;
    int L = seqlens[b];
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    const int n = (L + chunk - 1) / chunk;
    const float2 *ml = ws_ml + (size_t)bh * nsplit;
    float M = -INFINITY;
    for (int s = 0; s < n; ++s) M = fmaxf(M, ml[s].x);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f;
    for (int s = 0; s < n; ++s) Ls = fmaf(ex2(ml[s].x - Mu), ml[s].y, Ls);
    const float inv = (n > 0 && Ls > 0.f) ? 1.f / Ls : 0.f;
    const float *po = ws_o + (size_t)bh * nsplit * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float a = 0.f;
        for (int s = 0; s < n; ++s) a = fmaf(ex2(ml[s].x - Mu), po[(size_t)s * D + d], a);
        const float r = a * inv;
        if (OUT_F32)
            static_cast<float *>(o)[(size_t)bh * D + d] = r;
        else
            static_cast<__nv_bfloat16 *>(o)[(size_t)bh * D + d] = __float2bfloat16_rn(r);
    }
    if (lse != nullptr && threadIdx.x == 0)
        lse[bh] = (n > 0 && Ls > 0.f) ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
}

template <int D, int HG>
cudaError_t launch_split_t(const DecodeArgs &a, cudaStream_t st)
{
    constexpr int U = (HG >= 8) ? 2 : 4;
    const int G = a.Hq / a.Hkv;
    dim3 grid(a.nsplit, a.Hkv * (G / HG), a.B);
    decode_split_kernel<D, HG, U><<<grid, kSplitThreads, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.kc),
        static_cast<const __nv_bfloat16 *>(a.vc), a.seqlens, a.ws_o, a.ws_ml, a.Hq, a.Hkv,
        a.max_len, a.chunk, a.nsplit, a.scale_log2, a.status);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_split_d(const DecodeArgs &a, cudaStream_t st)
{
    const int G = a.Hq / a.Hkv;
    if (G % 8 == 0) return launch_split_t<D, 8>(a, st);
    if (G % 4 == 0) return launch_split_t<D, 4>(a, st);
    if (G % 2 == 0) return launch_split_t<D, 2>(a, st);
    return launch_split_t<D, 1>(a, st);
}

}  // namespace

int decode_chunk_len(int B, int Hkv, int max_len)
{
    // Aim for about four blocks per SM on a 152-SM GB300 at the shape's largest length;
    // chunks stay between 32 and 1024 keys.
    const long long target = 4LL * 152;
    int chunk = 1024;
    while (chunk > 32 &&
           (long long)B * Hkv * (((long long)max_len + chunk - 1) / chunk) < target)
        chunk /= 2;
    return chunk;
}

size_t decode_workspace_bytes(int B, int Hq, int D, int max_len, int chunk)
{
    const size_t nsplit = ((size_t)max_len + chunk - 1) / chunk;
    const size_t rows = (size_t)B * Hq * nsplit;
    return rows * D * sizeof(float) + rows * sizeof(float2);
}

cudaError_t launch_decode(const DecodeArgs &a, bool out_f32, cudaStream_t st)
{
    cudaError_t e = (a.D == 128) ? launch_split_d<128>(a, st) : launch_split_d<64>(a, st);
    if (e != cudaSuccess) return e;
    const int threads = a.D < 128 ? a.D : 128;
    if (out_f32)
        decode_merge_kernel<true><<<a.B * a.Hq, threads, 0, st>>>(
            a.ws_o, a.ws_ml, a.seqlens, a.o, a.lse, a.Hq, a.D, a.max_len, a.chunk, a.nsplit);
    else
        decode_merge_kernel<false><<<a.B * a.Hq, threads, 0, st>>>(
            a.ws_o, a.ws_ml, a.seqlens, a.o, a.lse, a.Hq, a.D, a.max_len, a.chunk, a.nsplit);
    return cudaGetLastError();
}

}  // namespace gqa
