// prefill_f32.cu -- fused attention forward in fp32 on CUDA cores (fp32 inputs and output).
//
// The fp32 entry point promises results within about 1e-5 of exact arithmetic, which rules
// out the tensor cores' reduced-precision fp32 (tf32) path; every product and sum here is an
// IEEE fp32 FMA/FADD (packed two at a time) and every exponential an fp32 expf.
//
// Structure (one thread block = 16 query rows of one head, 128 threads):
//   K and V tiles of KG x BN keys are staged in shared memory by asynchronous 16-byte copies,
//   two tiles in flight; key group kg takes keys [BN kg, BN kg + BN) of every tile, so each
//   row's keys are shared among KG independent sets of threads. Within a key group, 8 threads
//   share RT rows: thread t holds the head dims 32c + 4t .. 32c + 4t + 3 of each of its rows,
//   so every 16-byte vector read from shared memory serves RT rows (the shared-memory reads,
//   not the FMAs, bound a one-row-per-thread layout). BN = 8; head dim 64: RT = 4, KG = 4;
//   head dim 128: RT = 2, KG = 2.
//   For every 8 keys each thread forms 8 partial dot products per row; three halving
//   exchanges between the row's threads leave thread t with the full score of key 8i + t, so
//   each score is scaled, masked and exponentiated once, by one thread. The online-softmax
//   update per tile: m_new = max(m, tile max), c = exp(m - m_new), l = l c + sum exp(s - m_new),
//   acc = acc c + sum exp(s - m_new) v, with each probability passed to the row's other
//   threads for the P V product. At the end the key groups' (m, l, acc) are combined through
//   shared memory with weights exp(m_g - max_g m_g) (the same rescale, applied once more), then
//   O = acc / l and LSE = m + log l.
// Sources: "Attention three-op fusion" (xdnf.cn/news/349386) sections 2.2-2.3 (recurrence),
// 4.1-4.2 (K/V blocks staged in shared memory, output accumulator distributed over threads in
// registers, two block-wide synchronisations per tile), 4.3 (causal mask and fully masked
// tiles skipped), 6.1 (tail tile: out-of-range loads are 0 and their scores -inf).
#include "internal.h"
#include "ptx.cuh"

#include <cmath>

namespace gqa {
namespace {

constexpr int kTPR = 8;         // threads per row group (and keys per exchange)
constexpr int kRows = 16;       // query rows per block
constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct F32Cfg {
    static constexpr int RT = D == 64 ? 4 : 2;          // rows per thread
    static constexpr int KG = D == 64 ? 4 : 2;          // key groups
    static constexpr int BN = 8;                        // keys per key group and tile
    static constexpr int R = kRows;                     // query rows per block
    static constexpr int NT = R / RT * kTPR;            // threads per key group
    static constexpr int THREADS = KG * NT;             // 128 for both head dims
    static constexpr int SK = KG * BN;                  // keys per staged tile
    static constexpr int TILE = SK * D;                 // floats of K (or V) per tile
    static constexpr int SMEM = 2 * 2 * TILE * 4;       // two tiles of K and V, bytes
    static constexpr int NE = RT * (D / kTPR + 2);      // combine record per thread
    static_assert((KG - 1) * NE * NT * 4 <= SMEM, "combine records fit the tile buffers");
    static_assert(NT % 32 == 0 && BN % kTPR == 0 && D % (4 * kTPR) == 0, "shape");
};

__device__ __forceinline__ void cp_async16(void *sdst, const void *gsrc)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(sdst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Thread t of a group of kTPR lanes holds partial sums v[0..kTPR) (one per key); returns the
// sum over the group of v[t]. Each round halves the values a thread keeps: the thread with
// bit w of t set keeps the upper half and sends the lower half to its partner, and vice versa.
__device__ __forceinline__ float halving_exchange(float (&v)[kTPR], int t)
{
#pragma unroll
    for (int w = kTPR / 2; w >= 1; w /= 2) {
        const bool up = (t & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float keep = up ? v[w + j] : v[j];
            const float send = up ? v[j] : v[w + j];
            v[j] = keep + __shfl_xor_sync(kFull, send, w);
        }
    }
    return v[0];
}

template <int D>
__global__ void __launch_bounds__(F32Cfg<D>::THREADS, 4)
    prefill_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                       const float *__restrict__ v, float *__restrict__ o, float *__restrict__ lse,
                       int S, int Hq, int Hkv, float scale, int causal)
{
    using C = F32Cfg<D>;
    constexpr int RT = C::RT, NT = C::NT;
    constexpr int NC = D / (4 * kTPR);  // 16-byte chunks per thread and row
    constexpr int NG = C::BN / kTPR;    // exchange groups per key group and tile
    constexpr int DT = D / kTPR;        // dims per thread and row
    extern __shared__ __align__(16) float smem[];  // [stage][K, V][TILE], then combine records

    const int nrb = (S + C::R - 1) / C::R;
    const int rb = causal ? (nrb - 1 - (int)blockIdx.x) : (int)blockIdx.x;  // long rows first
    const int h = blockIdx.y, b = blockIdx.z;
    const int g = h / (Hq / Hkv);
    const int r0 = rb * C::R;
    const int kg = (int)threadIdx.x / NT;  // key group (whole warps)
    const int i = (int)threadIdx.x % NT;
    const int lane = threadIdx.x & 31;
    const int t = lane & (kTPR - 1);
    const int row0 = r0 + (i / kTPR) * RT;  // this thread's rows: row0 .. row0 + RT - 1

    float2 qv[RT][2 * NC], acc[RT][2 * NC];
    float m[RT], lp[RT];  // lp: this thread's share of each row sum
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        const bool live = row0 + r < S;
        const float *qrow = q + (((size_t)b * Hq + h) * S + (live ? row0 + r : 0)) * D + 4 * t;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float4 x = live ? *reinterpret_cast<const float4 *>(qrow + 4 * kTPR * c)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            qv[r][2 * c] = make_float2(x.x, x.y);
            qv[r][2 * c + 1] = make_float2(x.z, x.w);
            acc[r][2 * c] = acc[r][2 * c + 1] = make_float2(0.f, 0.f);
        }
        m[r] = -INFINITY;
        lp[r] = 0.f;
    }

    const float *kh = k + ((size_t)b * Hkv + g) * (size_t)S * D;
    const float *vh = v + ((size_t)b * Hkv + g) * (size_t)S * D;
    const int last_key = causal ? min(S - 1, r0 + C::R - 1) : S - 1;
    const int ntiles = last_key / C::SK + 1;

    auto stage = [&](int tile, int buf) {
        const int k0 = tile * C::SK;
        float *ks = smem + (size_t)buf * 2 * C::TILE, *vs = ks + C::TILE;
        for (int idx = threadIdx.x; idx < C::TILE / 4; idx += C::THREADS) {
            const int jj = idx / (D / 4), c4 = idx % (D / 4);
            float *kd = ks + jj * D + 4 * c4, *vd = vs + jj * D + 4 * c4;
            if (k0 + jj < S) {
                cp_async16(kd, kh + (size_t)(k0 + jj) * D + 4 * c4);
                cp_async16(vd, vh + (size_t)(k0 + jj) * D + 4 * c4);
            } else {
                *reinterpret_cast<float4 *>(kd) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(vd) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        cp_async_commit();
    };

    stage(0, 0);
    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        if (tile + 1 < ntiles) {
            stage(tile + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // this tile staged by every thread

        const float *Ks = smem + (size_t)buf * 2 * C::TILE + kg * C::BN * D;
        const float *Vs = Ks + C::TILE;
        const int k0 = tile * C::SK + kg * C::BN;
        float s[RT][NG];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            float part[RT][kTPR];
#pragma unroll
            for (int kk = 0; kk < kTPR; ++kk) {
                const float4 *kr =
                    reinterpret_cast<const float4 *>(Ks + (kTPR * gi + kk) * D) + t;
                float4 x[NC];
#pragma unroll
                for (int c = 0; c < NC; ++c) x[c] = kr[kTPR * c];
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        d2 = ffma2(qv[r][2 * c], make_float2(x[c].x, x[c].y), d2);
                        d2 = ffma2(qv[r][2 * c + 1], make_float2(x[c].z, x[c].w), d2);
                    }
                    part[r][kk] = d2.x + d2.y;
                }
            }
            const int key = k0 + kTPR * gi + t;
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                const float dot = halving_exchange(part[r], t);
                s[r][gi] = (key >= S || (causal && key > row0 + r)) ? -INFINITY : dot * scale;
            }
        }
        float p[RT][NG];
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            float tmax = s[r][0];
#pragma unroll
            for (int gi = 1; gi < NG; ++gi) tmax = fmaxf(tmax, s[r][gi]);
#pragma unroll
            for (int w = 1; w < kTPR; w *= 2) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, w));
            const float mn = fmaxf(m[r], tmax);
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            const float corr = expf(m[r] - mu);
            lp[r] *= corr;
            const float2 c2 = make_float2(corr, corr);
#pragma unroll
            for (int e = 0; e < 2 * NC; ++e) acc[r][e] = fmul2(acc[r][e], c2);
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                p[r][gi] = expf(s[r][gi] - mu);
                lp[r] += p[r][gi];
            }
            m[r] = mn;
        }
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
#pragma unroll
            for (int kk = 0; kk < kTPR; ++kk) {
                const float4 *vr =
                    reinterpret_cast<const float4 *>(Vs + (kTPR * gi + kk) * D) + t;
                float4 x[NC];
#pragma unroll
                for (int c = 0; c < NC; ++c) x[c] = vr[kTPR * c];
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    const float pk = __shfl_sync(kFull, p[r][gi], (lane & ~(kTPR - 1)) | kk);
                    const float2 p2 = make_float2(pk, pk);
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        acc[r][2 * c] = ffma2(p2, make_float2(x[c].x, x[c].y), acc[r][2 * c]);
                        acc[r][2 * c + 1] =
                            ffma2(p2, make_float2(x[c].z, x[c].w), acc[r][2 * c + 1]);
                    }
                }
            }
        }
        __syncthreads();  // every thread is done with this stage before it is refilled
    }

    // combine the key groups: groups 1.. post (acc, m, l) of each row in the now idle tile
    // buffers (element-major, so consecutive threads write consecutive words); group 0 merges
    if (C::KG > 1) {
        if (kg > 0) {
            float *w = smem + (size_t)(kg - 1) * C::NE * NT + i;
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                float *wr = w + (size_t)r * (DT + 2) * NT;
#pragma unroll
                for (int e = 0; e < 2 * NC; ++e) {
                    wr[(2 * e) * NT] = acc[r][e].x;
                    wr[(2 * e + 1) * NT] = acc[r][e].y;
                }
                wr[DT * NT] = m[r];
                wr[(DT + 1) * NT] = lp[r];
            }
        }
        __syncthreads();
        if (kg > 0) return;
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            const float *rr = smem + (size_t)r * (DT + 2) * NT + i;
            float M = m[r];
#pragma unroll
            for (int gg = 1; gg < C::KG; ++gg)
                M = fmaxf(M, rr[(size_t)(gg - 1) * C::NE * NT + DT * NT]);
            const float mu = (M == -INFINITY) ? 0.f : M;
            const float w0 = expf(m[r] - mu);
            lp[r] *= w0;
            const float2 w02 = make_float2(w0, w0);
#pragma unroll
            for (int e = 0; e < 2 * NC; ++e) acc[r][e] = fmul2(acc[r][e], w02);
#pragma unroll
            for (int gg = 1; gg < C::KG; ++gg) {
                const float *x = rr + (size_t)(gg - 1) * C::NE * NT;
                const float wg = expf(x[DT * NT] - mu);
                lp[r] = fmaf(wg, x[(DT + 1) * NT], lp[r]);
                const float2 wg2 = make_float2(wg, wg);
#pragma unroll
                for (int e = 0; e < 2 * NC; ++e)
                    acc[r][e] =
                        ffma2(wg2, make_float2(x[(2 * e) * NT], x[(2 * e + 1) * NT]), acc[r][e]);
            }
            m[r] = M;
        }
    }

#pragma unroll
    for (int r = 0; r < RT; ++r) {
        float l = lp[r];
#pragma unroll
        for (int w = 1; w < kTPR; w *= 2) l += __shfl_xor_sync(kFull, l, w);
        const int row = row0 + r;
        if (row < S) {
            float *orow = o + (((size_t)b * Hq + h) * S + row) * D + 4 * t;
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < NC; ++c)
                *reinterpret_cast<float4 *>(orow + 4 * kTPR * c) =
                    make_float4(acc[r][2 * c].x * inv, acc[r][2 * c].y * inv,
                                acc[r][2 * c + 1].x * inv, acc[r][2 * c + 1].y * inv);
            if (lse != nullptr && t == 0)
                lse[((size_t)b * Hq + h) * S + row] = l > 0.f ? m[r] + logf(l) : -INFINITY;
        }
    }
}

template <int D>
cudaError_t launch_f32(const float *q, const float *k, const float *v, float *o, float *lse,
                       int B, int S, int Hq, int Hkv, float scale, int causal, cudaStream_t st)
{
    using C = F32Cfg<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(prefill_f32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set[dev] = true;
    }
    dim3 grid((S + C::R - 1) / C::R, Hq, B);
    prefill_f32_kernel<D><<<grid, C::THREADS, C::SMEM, st>>>(q, k, v, o, lse, S, Hq, Hkv, scale,
                                                           causal);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, float *o,
                               float *lse, int B, int S, int Hq, int Hkv, int D, float scale,
                               int causal, cudaStream_t st)
{
    if (D == 64) return launch_f32<64>(q, k, v, o, lse, B, S, Hq, Hkv, scale, causal, st);
    return launch_f32<128>(q, k, v, o, lse, B, S, Hq, Hkv, scale, causal, st);
}

}  // namespace gqa
