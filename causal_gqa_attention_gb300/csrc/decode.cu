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

constexpr int kWarps = 4;  // consumer warps per block; each streams its own stages
constexpr int kRing = 2;   // stages in flight per warp

// Compile-time plan of the split kernel for head dim D and HG query heads per block.
template <int D, int HG>
struct Plan {
    static constexpr int LPK = D / 8;     // lanes per key row (8 dims = 16 bytes each)
    static constexpr int GPW = 32 / LPK;  // key groups per warp
    static constexpr int T = HG >= 8 ? 4 : (HG == 4 ? 8 : 16);  // keys per group per stage
    static constexpr int TG = T * HG;     // partial scores per lane before the reduction
    static constexpr int NV = TG / LPK;   // full scores per lane after it
    static constexpr int SK = GPW * T;    // keys per stage
    static constexpr int ROW = D * 2;     // bytes per K or V row
    static constexpr int STAGE = SK * ROW * 2;             // K rows, then V rows
    static constexpr int RING = kWarps * kRing * STAGE;
    static constexpr int PBUF = kWarps * GPW * T * HG * 8; // {p, p} per (key, head)
    static constexpr int COMB = kWarps * GPW * HG * (D + 2) * 4;
    static constexpr int BARS = kWarps * kRing * 8;
    static constexpr int SMEM = (RING > COMB ? RING : COMB) + PBUF + BARS;
    static_assert(TG % LPK == 0 && NV >= 1, "plan");
};

// One block per (key chunk, kv head, query-head subgroup, sequence), 4 warps. Each warp takes
// every 4th stage of SK keys of the chunk, copies its K and V rows into its own 2-stage ring
// with 1-D bulk copies (many bytes in flight, no registers held), and keeps an online-softmax
// state per key group: GPW groups of LPK lanes, a lane holding 8 of the D dims.
// Scores: each lane accumulates partial dot products for T keys x HG heads over its 8 dims
// (packed fp32 pairs), then the LPK lanes of a group reduce them by halving exchanges, after
// which lane gl holds the complete scores of entries gl*NV .. gl*NV+NV-1 (entry = t*HG + h).
// The running max per head is rescaled lazily (only when a score exceeds it by 2^8), the
// probabilities go through shared memory to the lanes that own the V dims, and P V uses
// packed fp32 FMAs.
template <int D, int HG>
__global__ void __launch_bounds__(kWarps * 32)
    decode_split_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kc,
                        const __nv_bfloat16 *__restrict__ vc, const int *__restrict__ seqlens,
                        float *__restrict__ ws_o, float2 *__restrict__ ws_ml, int Hq, int Hkv,
                        int max_len, int chunk, int nsplit, float scale_log2,
                        unsigned *__restrict__ status)
{
    using P = Plan<D, HG>;
    constexpr int LPK = P::LPK, GPW = P::GPW, T = P::T, TG = P::TG, NV = P::NV, SK = P::SK;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float2 *pbuf = reinterpret_cast<float2 *>(smem + (P::RING > P::COMB ? P::RING : P::COMB));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (P::RING > P::COMB ? P::RING : P::COMB) +
                                                  P::PBUF);
    float *comb = reinterpret_cast<float *>(smem);  // reuses the ring after the last stage

    const int split = blockIdx.x;
    const int subgroups = gridDim.y / Hkv;
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
    const int nstage = (end - start + SK - 1) / SK;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int grp = lane / LPK, gl = lane % LPK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWarps * kRing; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const size_t head_off = ((size_t)b * Hkv + g) * (size_t)max_len * D;
    const __nv_bfloat16 *kb = kc + head_off;
    const __nv_bfloat16 *vb = vc + head_off;
    auto issue = [&](int i) {  // stage i of the chunk into this warp's ring
        const int slot = (i / kWarps) % kRing;
        const int k0 = start + i * SK;
        const uint32_t n = (uint32_t)min(SK, end - k0);
        uint8_t *dst = ring + (warp * kRing + slot) * P::STAGE;
        uint64_t *bar = &bars[warp * kRing + slot];
        mbar_arrive_expect_tx(bar, 2u * n * P::ROW);
        bulk_load(dst, kb + (size_t)k0 * D, n * P::ROW, bar);
        bulk_load(dst + SK * P::ROW, vb + (size_t)k0 * D, n * P::ROW, bar);
    };
    if (lane == 0)
        for (int r = 0; r < kRing; ++r)
            if (warp + r * kWarps < nstage) issue(warp + r * kWarps);

    // query fragments (8 dims of each head), scaled so scores come out in log2 units
    float2 qp[HG][4];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        const uint4 w = *reinterpret_cast<const uint4 *>(q + ((size_t)b * Hq + h0 + h) * D + gl * 8);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            qp[h][e] = make_float2(bf16lo(ws[e]) * scale_log2, bf16hi(ws[e]) * scale_log2);
    }

    float m_ref[HG];       // running max reference per head (uniform over the group)
    float2 acc[HG][4];     // unnormalised output, this lane's 8 dims of each head
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        m_ref[h] = -INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
    }
    float l_own[NV];       // this lane's share of the running sums (entries it owns)
#pragma unroll
    for (int v = 0; v < NV; ++v) l_own[v] = 0.f;

    volatile int never = 0;
    bool ok = true;
    int it = 0;
    for (int i = warp; i < nstage; i += kWarps, ++it) {
        const int slot = it % kRing;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[warp * kRing + slot], (it / kRing) & 1, &never));
        if (!ok) break;
        const uint8_t *stage = ring + (warp * kRing + slot) * P::STAGE;
        const int k0 = start + i * SK;
        const int nvalid = min(SK, end - k0);

        // ---- partial scores for the T keys of this lane's group
        float part[TG];
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const uint4 w = *reinterpret_cast<const uint4 *>(stage + (grp * T + t) * P::ROW + gl * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            float2 kp[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) kp[e] = make_float2(bf16lo(ws[e]), bf16hi(ws[e]));
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 4; ++e) d2 = ffma2(qp[h][e], kp[e], d2);
                part[t * HG + h] = d2.x + d2.y;
            }
        }
        // ---- halving exchange across the LPK lanes of the group
#pragma unroll
        for (int off = LPK / 2, cur = TG; off >= 1; off >>= 1, cur >>= 1) {
            const bool up = (gl & off) != 0;
#pragma unroll
            for (int e = 0; e < cur / 2; ++e) {
                const float send = up ? part[e] : part[e + cur / 2];
                const float keep = up ? part[e + cur / 2] : part[e];
                part[e] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
        // part[v] is now the full score of entry gl*NV + v: key t = entry / HG, head entry % HG
        float mv[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int ent = gl * NV + v;
            const int t = ent / HG, hh = ent % HG;
            if (grp * T + t >= nvalid) part[v] = -INFINITY;
            float mr = m_ref[0];
#pragma unroll
            for (int h = 1; h < HG; ++h) mr = (hh == h) ? m_ref[h] : mr;
            mv[v] = mr;
        }
        bool need = false;
#pragma unroll
        for (int v = 0; v < NV; ++v) need |= part[v] > mv[v] + 8.0f;
        if (__any_sync(0xffffffffu, need)) {
            // exact block max per head over the group, then rescale to it
#pragma unroll
            for (int h = 0; h < HG; ++h) {
                float bm = -INFINITY;
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    if ((gl * NV + v) % HG == h) bm = fmaxf(bm, part[v]);
#pragma unroll
                for (int off = LPK / 2; off >= 1; off >>= 1)
                    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
                const float mn = fmaxf(m_ref[h], bm);
                if (mn > m_ref[h]) {
                    const float alpha = ex2(m_ref[h] - mn);  // 0 when m_ref was -inf
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[h][e] = fmul2(acc[h][e], a2);
#pragma unroll
                    for (int v = 0; v < NV; ++v)
                        if ((gl * NV + v) % HG == h) l_own[v] *= alpha;
                    m_ref[h] = mn;
                }
            }
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int hh = (gl * NV + v) % HG;
                float mr = m_ref[0];
#pragma unroll
                for (int h = 1; h < HG; ++h) mr = (hh == h) ? m_ref[h] : mr;
                mv[v] = mr;
            }
        }
        // ---- probabilities: own entries, then to shared memory for the V lanes
        float2 *pw = pbuf + (warp * GPW + grp) * T * HG;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const float mu = (mv[v] == -INFINITY) ? 0.f : mv[v];
            const float p = ex2(part[v] - mu);
            l_own[v] += p;
            pw[gl * NV + v] = make_float2(p, p);
        }
        __syncwarp();
        // ---- O += P V for the group's keys
#pragma unroll
        for (int t = 0; t < T; ++t) {
            if (grp * T + t < nvalid) {
                const uint4 w = *reinterpret_cast<const uint4 *>(stage + SK * P::ROW +
                                                                 (grp * T + t) * P::ROW + gl * 16);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                float2 vp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) vp[e] = make_float2(bf16lo(ws[e]), bf16hi(ws[e]));
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    const float2 pp = pw[t * HG + h];
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[h][e] = ffma2(pp, vp[e], acc[h][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && i + kRing * kWarps < nstage) {
            fence_proxy_async_smem();
            issue(i + kRing * kWarps);
        }
    }
    if (!ok) {
        // a stage never arrived: report, let this warp's copies land, and give up
        if (lane == 0) atomicOr(status, 2u);
        for (int r = 0; r < kRing; ++r) {
            const int i2 = warp + (it + r) * kWarps;
            if (i2 < nstage) mbar_wait(&bars[warp * kRing + (it + r) % kRing], ((it + r) / kRing) & 1, &never);
        }
    }

    // ---- running sums per head over the group's lanes
    float lsum[HG];
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        float x = 0.f;
#pragma unroll
        for (int v = 0; v < NV; ++v)
            if ((gl * NV + v) % HG == h) x += l_own[v];
#pragma unroll
        for (int off = LPK / 2; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        lsum[h] = x;
    }
    __syncthreads();  // every warp done with the ring: reuse it for the combine
    // comb layout: [state = warp*GPW + grp][h][D + 2]: D outputs, then m and l
    const int st = warp * GPW + grp;
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        float *row = comb + ((size_t)st * HG + h) * (D + 2);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            row[gl * 8 + 2 * e] = acc[h][e].x;
            row[gl * 8 + 2 * e + 1] = acc[h][e].y;
        }
        if (gl == 0) {
            row[D] = ok ? m_ref[h] : -INFINITY;
            row[D + 1] = ok ? lsum[h] : 0.f;
        }
    }
    __syncthreads();
    constexpr int NST = kWarps * GPW;
    for (int idx = threadIdx.x; idx < HG * D; idx += kWarps * 32) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
        for (int s2 = 0; s2 < NST; ++s2) M = fmaxf(M, comb[((size_t)s2 * HG + h) * (D + 2) + D]);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f, a = 0.f;
        for (int s2 = 0; s2 < NST; ++s2) {
            const float *row = comb + ((size_t)s2 * HG + h) * (D + 2);
            const float w = ex2(row[D] - Mu);
            Ls = fmaf(w, row[D + 1], Ls);
            a = fmaf(w, row[d], a);
        }
        const size_t orow = ((size_t)b * Hq + h0 + h) * nsplit + split;
        ws_o[orow * D + d] = a;
        if (d == 0) ws_ml[orow] = make_float2(M, Ls);
    }
    // the merge kernel may start launching once every block got here (or exited)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kMergeWarps = 4;  // (sequence, query head) rows per merge block, one per warp

// One warp per (sequence, query head): the chunk states are combined with weights
// 2^(m_s - M), M = max_s m_s, visiting the chunks in order (deterministic). Chunk states are
// read 32 at a time (one per lane) and their outputs with all loads issued before use; D/32
// dims per lane. Launched as a programmatic dependent of the split kernel: everything before
// the grid-dependency wait overlaps the split kernel's tail.
template <bool OUT_F32, int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    decode_merge_kernel(const float *__restrict__ ws_o, const float2 *__restrict__ ws_ml,
                        const int *__restrict__ seqlens, void *__restrict__ o,
                        float *__restrict__ lse, int BH, int Hq, int max_len, int chunk, int nsplit)
{
    constexpr int DL = D / 32;  // dims per lane
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x * kMergeWarps + warp;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (bh >= BH) return;
    const int b = bh / Hq;
    int L = seqlens[b];
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    const int n = (L + chunk - 1) / chunk;
    const float2 *ml = ws_ml + (size_t)bh * nsplit;
    const float *po = ws_o + (size_t)bh * nsplit * D + lane * DL;

    float M = -INFINITY, Ls = 0.f, acc[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = 0.f;
    for (int s0 = 0; s0 < n; s0 += 32) {
        const int cnt = min(32, n - s0);
        const float2 mine = lane < cnt ? ml[s0 + lane] : make_float2(-INFINITY, 0.f);
        float cm = mine.x;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
        const float Mn = fmaxf(M, cm);
        const float Mu = (Mn == -INFINITY) ? 0.f : Mn;
        const float w = ex2(mine.x - Mu);
        float cs = w * mine.y;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
        const float a = ex2(M - Mu);
        Ls = fmaf(Ls, a, cs);
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[e] *= a;
        for (int j0 = 0; j0 < cnt; j0 += 8) {
            float x[8][DL];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j0 + j < cnt) {
                    const float *src = po + (size_t)(s0 + j0 + j) * D;
                    if (DL == 4) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(src);
                        x[j][0] = v4.x; x[j][1] = v4.y; x[j][DL > 2 ? 2 : 0] = v4.z;
                        x[j][DL > 3 ? 3 : 0] = v4.w;
                    } else {
                        const float2 v2 = *reinterpret_cast<const float2 *>(src);
                        x[j][0] = v2.x; x[j][DL > 1 ? 1 : 0] = v2.y;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float wj = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
                if (j0 + j < cnt)
#pragma unroll
                    for (int e = 0; e < DL; ++e) acc[e] = fmaf(wj, x[j][e], acc[e]);
            }
        }
        M = Mn;
    }
    const float inv = (n > 0 && Ls > 0.f) ? 1.f / Ls : 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) {
        const float r = acc[e] * inv;
        if (OUT_F32)
            static_cast<float *>(o)[(size_t)bh * D + lane * DL + e] = r;
        else
            static_cast<__nv_bfloat16 *>(o)[(size_t)bh * D + lane * DL + e] = __float2bfloat16_rn(r);
    }
    if (lse != nullptr && lane == 0)
        lse[bh] = (n > 0 && Ls > 0.f) ? (M + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
}

template <bool OUT_F32, int D>
cudaError_t launch_merge(const DecodeArgs &a, cudaStream_t st)
{
    const int BH = a.B * a.Hq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((BH + kMergeWarps - 1) / kMergeWarps);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<OUT_F32, D>, (const float *)a.ws_o,
                              (const float2 *)a.ws_ml, a.seqlens, a.o, a.lse, BH, a.Hq, a.max_len,
                              a.chunk, a.nsplit);
}

template <int D, int HG>
cudaError_t launch_split_t(const DecodeArgs &a, cudaStream_t st)
{
    using P = Plan<D, HG>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_split_kernel<D, HG>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set[dev] = true;
    }
    const int G = a.Hq / a.Hkv;
    dim3 grid(a.nsplit, a.Hkv * (G / HG), a.B);
    decode_split_kernel<D, HG><<<grid, kWarps * 32, P::SMEM, st>>>(
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
    // Aim for about three blocks per SM on a 152-SM GB300 at the shape's largest length;
    // chunks stay between 64 and 512 keys (at least one stage per warp of a block).
    const long long target = 3LL * 152;
    int chunk = 512;
    while (chunk > 64 &&
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
    if (a.D == 128)
        e = out_f32 ? launch_merge<true, 128>(a, st) : launch_merge<false, 128>(a, st);
    else
        e = out_f32 ? launch_merge<true, 64>(a, st) : launch_merge<false, 64>(a, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gqa
