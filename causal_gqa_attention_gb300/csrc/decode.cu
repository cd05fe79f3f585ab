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
// Online-softmax update of one group's state with one stage (T keys per group, nvalid valid
// keys in the stage). K rows of the stage first, V rows after them. Lane gl of group grp holds
// dims gl*8 .. gl*8+7; `pw` is this group's {p, p} buffer in shared memory.
template <int D, int HG>
__device__ __forceinline__ void stage_update(const uint8_t *stage, int nvalid, int grp, int gl,
                                             const float2 (&qp)[HG][4], float (&m_ref)[HG],
                                             float2 (&acc)[HG][4],
                                             float (&l_own)[Plan<D, HG>::NV], float2 *pw)
{
    using P = Plan<D, HG>;
    constexpr int LPK = P::LPK, T = P::T, TG = P::TG, NV = P::NV, SK = P::SK;
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
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const float mu = (mv[v] == -INFINITY) ? 0.f : mv[v];
        const float p = ex2(part[v] - mu);
        l_own[v] += p;
        pw[gl * NV + v] = make_float2(p, p);
    }
    __syncwarp();
    // ---- O += P V for the group's keys. V rows past nvalid are zero (the split kernel clears
    // its ring at start, the stream kernel clears them before a partial stage's copy) and get
    // p = 0.
#pragma unroll
    for (int t = 0; t < T; ++t) {
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
    __syncwarp();
}

// Running sums per head over the LPK lanes of a group (each lane holds the sums of its entries).
template <int D, int HG>
__device__ __forceinline__ void group_sums(const float (&l_own)[Plan<D, HG>::NV], int gl,
                                           float (&lsum)[HG])
{
    using P = Plan<D, HG>;
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        float x = 0.f;
#pragma unroll
        for (int v = 0; v < P::NV; ++v)
            if ((gl * P::NV + v) % HG == h) x += l_own[v];
#pragma unroll
        for (int off = P::LPK / 2; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        lsum[h] = x;
    }
}

// q fragment (8 dims of each of the HG heads starting at h0), scaled to log2 units. q is bf16,
// or fp32 when it comes from the RoPE step (kept unrounded).
template <int D, int HG, typename QT>
__device__ __forceinline__ void load_q(const QT *q, size_t row0, int gl, float scale_log2,
                                       float2 (&qp)[HG][4])
{
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        if constexpr (sizeof(QT) == 4) {
            const float4 *src = reinterpret_cast<const float4 *>(q + (row0 + h) * D + gl * 8);
            const float4 a = src[0], c = src[1];
            qp[h][0] = make_float2(a.x * scale_log2, a.y * scale_log2);
            qp[h][1] = make_float2(a.z * scale_log2, a.w * scale_log2);
            qp[h][2] = make_float2(c.x * scale_log2, c.y * scale_log2);
            qp[h][3] = make_float2(c.z * scale_log2, c.w * scale_log2);
        } else {
            const uint4 w = *reinterpret_cast<const uint4 *>(q + (row0 + h) * D + gl * 8);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                qp[h][e] = make_float2(bf16lo(ws[e]) * scale_log2, bf16hi(ws[e]) * scale_log2);
        }
    }
}

// RoPE for decode (rotate-half): the pair (d, d + D/2) becomes
// [x1 cos - x2 sin, x1 sin + x2 cos] with the angle tables' row of the token's position. Lane gl
// of a key group holds dims gl*8 .. gl*8+7; the partner half sits LPK/2 lanes away, so one
// exchange gives every lane both halves of its 8 pairs. cs / sn point at the tables' row.
// The table entries this lane needs: pairs (gl % HALF) * 8 .. + 7 of the row.
template <int D>
__device__ __forceinline__ void rope_angles(int gl, const float *cs, const float *sn,
                                            float (&c)[8], float (&sv)[8])
{
    constexpr int HALF = D / 16;  // LPK / 2
    const int i0 = (gl % HALF) * 8;
    const float4 c0 = *reinterpret_cast<const float4 *>(cs + i0);
    const float4 c1 = *reinterpret_cast<const float4 *>(cs + i0 + 4);
    const float4 s0 = *reinterpret_cast<const float4 *>(sn + i0);
    const float4 s1 = *reinterpret_cast<const float4 *>(sn + i0 + 4);
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
    c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    sv[0] = s0.x; sv[1] = s0.y; sv[2] = s0.z; sv[3] = s0.w;
    sv[4] = s1.x; sv[5] = s1.y; sv[6] = s1.z; sv[7] = s1.w;
}

template <int D>
__device__ __forceinline__ void rope_rotate8(float (&x)[8], int gl, const float (&c)[8],
                                             const float (&sv)[8])
{
    constexpr int HALF = D / 16;
    const bool upper = gl >= HALF;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, x[e], HALF);
        x[e] = upper ? other * sv[e] + x[e] * c[e] : x[e] * c[e] - other * sv[e];
    }
}

// Eight bf16 values of one row, widened to fp32.
__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16 *src, float (&x)[8])
{
    const uint4 w = *reinterpret_cast<const uint4 *>(src);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = bf16lo(ws[e]);
        x[2 * e + 1] = bf16hi(ws[e]);
    }
}

// q fragment as load_q, rotated by RoPE first (in fp32, never rounded).
template <int D, int HG>
__device__ __forceinline__ void load_q_rope(const __nv_bfloat16 *q, size_t row0, int gl,
                                            float scale_log2, const float (&c)[8],
                                            const float (&sv)[8], float2 (&qp)[HG][4])
{
#pragma unroll
    for (int h = 0; h < HG; ++h) {
        float x[8];
        load_bf16x8(q + (row0 + h) * D + gl * 8, x);
        rope_rotate8<D>(x, gl, c, sv);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            qp[h][e] = make_float2(x[2 * e] * scale_log2, x[2 * e + 1] * scale_log2);
    }
}

// The new token's K/V for decode with RoPE (unrotated key, value, angle tables, and the cache
// to store the rotated key and the value in). Unused (null) in plain decode.
struct RopeIn {
    const __nv_bfloat16 *k_new, *v_new;  // [B, Hkv, D]
    const float *cos_t, *sin_t;          // [max_len, D/2]
    __nv_bfloat16 *kc, *vc;              // the caches, written at row seqlens[b] - 1
};

template <int D, int HG, typename QT>
__global__ void __launch_bounds__(kWarps * 32)
    decode_split_kernel(const QT *__restrict__ q, const __nv_bfloat16 *__restrict__ kc,
                        const __nv_bfloat16 *__restrict__ vc, const int *__restrict__ seqlens,
                        float *__restrict__ ws_o, float2 *__restrict__ ws_ml, int Hq, int Hkv,
                        int max_len, int chunk, int nsplit, float scale_log2,
                        unsigned *__restrict__ status, long long wait_limit)
{
    using P = Plan<D, HG>;
    constexpr int LPK = P::LPK, GPW = P::GPW, T = P::T, NV = P::NV, SK = P::SK;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float2 *pbuf = reinterpret_cast<float2 *>(smem + (P::RING > P::COMB ? P::RING : P::COMB));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (P::RING > P::COMB ? P::RING : P::COMB) +
                                                  P::PBUF);
    float *comb = reinterpret_cast<float *>(smem);  // reuses the ring after the last stage

    // launched as a programmatic dependent: nothing from global memory is read before the
    // previous kernel in the stream has finished and flushed
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

    for (int i = threadIdx.x; i < P::RING / 16; i += kWarps * 32)
        reinterpret_cast<uint4 *>(ring)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
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
        if (!dbg_ok(n >= 1 && k0 + (int)n <= max_len, status)) {
            mbar_arrive(bar);  // nothing copied: the stage completes empty
            return;
        }
        mbar_arrive_expect_tx(bar, 2u * n * P::ROW);
        bulk_load(dst, kb + (size_t)k0 * D, n * P::ROW, bar);
        bulk_load(dst + SK * P::ROW, vb + (size_t)k0 * D, n * P::ROW, bar);
    };
    if (lane == 0)
        for (int r = 0; r < kRing; ++r)
            if (warp + r * kWarps < nstage) issue(warp + r * kWarps);

    float2 qp[HG][4];
    load_q<D, HG, QT>(q, (size_t)b * Hq + h0, gl, scale_log2, qp);

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
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[warp * kRing + slot], (it / kRing) & 1, &never, wait_limit));
        if (!ok) break;
        const uint8_t *stage = ring + (warp * kRing + slot) * P::STAGE;
        const int k0 = start + i * SK;
        const int nvalid = min(SK, end - k0);

        stage_update<D, HG>(stage, nvalid, grp, gl, qp, m_ref, acc, l_own,
                            pbuf + (warp * GPW + grp) * T * HG);
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
            if (i2 < nstage)
                mbar_wait_drain(&bars[warp * kRing + (it + r) % kRing], ((it + r) / kRing) & 1);
        }
    }

    float lsum[HG];
    group_sums<D, HG>(l_own, gl, lsum);
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
        if (!dbg_ok(orow < (size_t)gridDim.z * Hq * nsplit, status)) continue;
        ws_o[orow * D + d] = a;
        if (d == 0) ws_ml[orow] = make_float2(M, Ls);
    }
    // the merge kernel may start launching once every block got here (or exited)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ stream split (B <= 1024)

constexpr int kStreamMaxWarps = 1824;  // 152 SMs x 3 resident blocks x 4 warps
// Smallest slice of keys a warp is given: one fill of its 2-stage ring of 16-key stages. Small
// calls then spread over as many warps as that allows, each with a single round of copies
// (B1 L4096: 14.3 us one call, 10.4 us back to back, against 16.4 / 11.9 us with 64-key slices
// and 16.4 / 11.4 us with 16-key slices, whose pieces double the merge's reads).
constexpr int kStreamMinKeys = 32;
constexpr int kStreamMaxBatch = 1024;  // larger batches use the chunked kernel

__device__ __forceinline__ int clamp_len(int L, int max_len)
{
    return L < 0 ? 0 : (L > max_len ? max_len : L);
}

// Sum over b in [0, nb) of clamp(seqlens[b]), over the warp (every lane gets the total).
__device__ __forceinline__ long long warp_len_sum(const int *seqlens, int nb, int max_len, int lane)
{
    long long x = 0;
    for (int b = lane; b < nb; b += 32) x += clamp_len(seqlens[b], max_len);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// The keys of all sequences and all (kv head, query-head subgroup) streams form one list:
// sequence b, stream s_local (NGS per sequence), key j at position
//   NGS * sum_{b' < b} L_b' + s_local * L_b + j.
// Warp W of the NWT warps of the grid takes positions [W*KP, W*KP + KP) with
// KP = max(ceil(total / NWT), kStreamMinKeys): every warp moves the same number of bytes.
// Where a slice crosses a stream boundary it produces one partial per piece; piece
// (warp W, stream s = b*NGS + s_local) is stored at index W + s (unique, since both grow
// along the list), so the merge finds the pieces of a stream as a contiguous range of warps.
__device__ __forceinline__ long long stream_slice(long long total, int nwt)
{
    const long long kp = (total + nwt - 1) / nwt;
    return kp > kStreamMinKeys ? kp : (long long)kStreamMinKeys;
}

struct StreamCursor {
    long long pos;  // list position of the next key
    int b, sl, off, Lb;
};

__device__ __forceinline__ void cursor_advance(StreamCursor &c, int n, const int *seqlens, int B,
                                               int max_len, int NGS)
{
    c.pos += n;
    c.off += n;
    if (c.off == c.Lb) {
        c.off = 0;
        if (++c.sl == NGS) {
            c.sl = 0;
            do {
                ++c.b;
                c.Lb = c.b < B ? clamp_len(seqlens[c.b], max_len) : 0;
            } while (c.b < B && c.Lb == 0);
        }
    }
}

// ROPE: the step also applies RoPE to q and to the new key at position seqlens[b] - 1 and
// stores the new key and value in the cache. The warp whose stage holds that row (the last key
// of a stream) replaces the row in shared memory (it was loaded before the store) with the
// rotated key, rounded to bf16 as the cache holds it, and the value; the stream of query-head
// subgroup 0 of each kv head also writes them to the cache.
template <int D, int HG, bool ROPE>
__global__ void __launch_bounds__(kWarps * 32)
    decode_stream_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ kc,
                         const __nv_bfloat16 *__restrict__ vc, const int *__restrict__ seqlens,
                         float *__restrict__ ws_o, float2 *__restrict__ ws_ml, int B, int Hq,
                         int Hkv, int max_len, float scale_log2, unsigned *__restrict__ status,
                         RopeIn rope, long long wait_limit)
{
    using P = Plan<D, HG>;
    constexpr int LPK = P::LPK, GPW = P::GPW, T = P::T, NV = P::NV, SK = P::SK;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float2 *pbuf = reinterpret_cast<float2 *>(smem + P::RING);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::RING + P::PBUF);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int grp = lane / LPK, gl = lane % LPK;
    const int G = Hq / Hkv, SUB = G / HG, NGS = Hkv * SUB;
    const int W = blockIdx.x * kWarps + warp, NWT = gridDim.x * kWarps;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWarps * kRing; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // launched as a programmatic dependent: nothing from global memory is read before the
    // previous kernel in the stream has finished and flushed
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- this warp's slice of the key list
    bool bad = false;
    for (int b = lane; b < B; b += 32) {
        const int L = seqlens[b];
        bad |= (L < 0 || L > max_len);
    }
    if (__any_sync(0xffffffffu, bad) && W == 0 && lane == 0) atomicOr(status, 1u);
    const long long total = warp_len_sum(seqlens, B, max_len, lane) * NGS;
    const long long KP = stream_slice(total, NWT);
    const long long r0 = (long long)W * KP;
    const long long r1 = r0 + KP < total ? r0 + KP : total;
    if (r0 < total) {
        // sequence holding position r0: scan the per-sequence list lengths 32 at a time
        long long base = 0;
        int b = 0;
        for (int b0 = 0;; b0 += 32) {
            const int bb = b0 + lane;
            const long long x = bb < B ? (long long)clamp_len(seqlens[bb], max_len) * NGS : 0;
            long long incl = x;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const long long tot32 = __shfl_sync(0xffffffffu, incl, 31);
            if (r0 < base + tot32) {
                const unsigned m = __ballot_sync(0xffffffffu, base + incl > r0);
                const int j = __ffs(m) - 1;
                b = b0 + j;
                base += __shfl_sync(0xffffffffu, incl - x, j);
                break;
            }
            base += tot32;
        }
        StreamCursor c0;
        c0.pos = r0;
        c0.b = b;
        c0.Lb = clamp_len(seqlens[b], max_len);
        const long long rel = r0 - base;
        c0.sl = (int)(rel / c0.Lb);
        c0.off = (int)(rel % c0.Lb);

        // ---- producer side (lane 0 issues; every lane tracks the cursor)
        StreamCursor pc = c0;
        int issued = 0;
        auto issue_next = [&]() {
            if (pc.pos >= r1) return;
            const long long left_piece = (long long)(pc.Lb - pc.off);
            const long long left_slice = r1 - pc.pos;
            const int n = (int)min((long long)SK, min(left_piece, left_slice));
            const int slot = issued % kRing;
            uint8_t *dst = ring + (warp * kRing + slot) * P::STAGE;
            if (n < SK) {
                // V rows past the copy get p = 0, and 0 * NaN would not be 0: zero them (the
                // ring is not cleared at start, and a slot keeps an earlier stage's rows)
                uint4 *vz = reinterpret_cast<uint4 *>(dst + (SK + n) * P::ROW);
                for (int c = lane; c < (SK - n) * P::ROW / 16; c += 32) vz[c] = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                const int g = pc.sl / SUB;
                const size_t row = ((size_t)pc.b * Hkv + g) * (size_t)max_len + pc.off;
                uint64_t *bar = &bars[warp * kRing + slot];
                if (dbg_ok(pc.b < B && g < Hkv && n >= 1 && pc.off + n <= max_len, status)) {
                    mbar_arrive_expect_tx(bar, 2u * n * P::ROW);
                    bulk_load(dst, kc + row * D, n * P::ROW, bar);
                    bulk_load(dst + SK * P::ROW, vc + row * D, n * P::ROW, bar);
                } else {
                    mbar_arrive(bar);  // nothing copied: the stage completes empty
                }
            }
            cursor_advance(pc, n, seqlens, B, max_len, NGS);
            ++issued;
        };
        for (int r = 0; r < kRing; ++r) issue_next();

        // ---- consumer side
        StreamCursor cc = c0;
        float2 qp[HG][4];
        float m_ref[HG];
        float2 acc[HG][4];
        float l_own[NV];
        uint4 new_k = make_uint4(0, 0, 0, 0), new_v = new_k;  // RoPE: the new row, packed bf16
        float2 *pw = pbuf + (warp * GPW + grp) * T * HG;
        volatile int never = 0;
        int it = 0;
        bool ok = true;
        while (cc.pos < r1) {
            const int n = (int)min((long long)SK, min((long long)(cc.Lb - cc.off), r1 - cc.pos));
            const bool first = (cc.pos == r0) || (cc.off == 0);
            const bool last = (cc.off + n == cc.Lb) || (cc.pos + n == r1);
            if (first) {
                const int g = cc.sl / SUB, gs = cc.sl % SUB;
                if constexpr (ROPE) {
                    // angles of the newest token's position, for q and (when this slice ends
                    // the stream) for the new key, which is rotated and packed here so the
                    // stage that holds its row needs no global load
                    const size_t prow = (size_t)(cc.Lb - 1) * (D / 2);
                    float c[8], sv[8];
                    rope_angles<D>(gl, rope.cos_t + prow, rope.sin_t + prow, c, sv);
                    load_q_rope<D, HG>(q, (size_t)cc.b * Hq + g * G + gs * HG, gl, scale_log2,
                                       c, sv, qp);
                    if (cc.pos + (cc.Lb - cc.off) <= r1) {
                        const size_t src = ((size_t)cc.b * Hkv + g) * D + gl * 8;
                        float x[8];
                        load_bf16x8(rope.k_new + src, x);
                        rope_rotate8<D>(x, gl, c, sv);
                        new_k = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                           pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
                        new_v = *reinterpret_cast<const uint4 *>(rope.v_new + src);
                    }
                } else {
                    load_q<D, HG, __nv_bfloat16>(q, (size_t)cc.b * Hq + g * G + gs * HG, gl,
                                                 scale_log2, qp);
                }
#pragma unroll
                for (int h = 0; h < HG; ++h) {
                    m_ref[h] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int v = 0; v < NV; ++v) l_own[v] = 0.f;
            }
            const int slot = it % kRing;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars[warp * kRing + slot], (it / kRing) & 1, &never, wait_limit));
            if (!ok) break;
            if constexpr (ROPE) {
                if (cc.off + n == cc.Lb) {  // the stage holds the newest key, as its row n - 1
                    const int g = cc.sl / SUB;
                    const uint4 kw = new_k, vw = new_v;
                    if (grp == 0) {
                        uint8_t *stg = ring + (warp * kRing + slot) * P::STAGE;
                        *reinterpret_cast<uint4 *>(stg + (n - 1) * P::ROW + gl * 16) = kw;
                        *reinterpret_cast<uint4 *>(stg + (SK + n - 1) * P::ROW + gl * 16) = vw;
                        if (cc.sl % SUB == 0) {
                            const size_t row =
                                (((size_t)cc.b * Hkv + g) * max_len + (cc.Lb - 1)) * D + gl * 8;
                            *reinterpret_cast<uint4 *>(rope.kc + row) = kw;
                            *reinterpret_cast<uint4 *>(rope.vc + row) = vw;
                        }
                    }
                    __syncwarp();
                }
            }
            stage_update<D, HG>(ring + (warp * kRing + slot) * P::STAGE, n, grp, gl, qp, m_ref,
                                acc, l_own, pw);
            if (last) {
                float lsum[HG];
                group_sums<D, HG>(l_own, gl, lsum);
                // combine the GPW groups of the warp (lanes gl, gl + LPK, ...)
#pragma unroll
                for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
                    for (int h = 0; h < HG; ++h) {
                        const float mo = __shfl_xor_sync(0xffffffffu, m_ref[h], off);
                        const float mn = fmaxf(m_ref[h], mo);
                        const float mu = (mn == -INFINITY) ? 0.f : mn;
                        const float a = ex2(m_ref[h] - mu);
                        lsum[h] *= a;
                        lsum[h] += __shfl_xor_sync(0xffffffffu, lsum[h], off);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[h][e] = fmul2(acc[h][e], make_float2(a, a));
                            acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, off);
                            acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, off);
                        }
                        m_ref[h] = mn;
                    }
                }
                // piece (warp W, stream s) is row W + s of at most NWT + B * NGS
                if (grp == 0 &&
                    dbg_ok((size_t)W + (size_t)cc.b * NGS + cc.sl < (size_t)NWT + (size_t)B * NGS,
                           status)) {
                    const size_t piece = (size_t)W + (size_t)cc.b * NGS + cc.sl;
#pragma unroll
                    for (int h = 0; h < HG; ++h) {
                        float4 *dst = reinterpret_cast<float4 *>(ws_o + (piece * HG + h) * D + gl * 8);
                        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
                        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
                        if (gl == 0) ws_ml[piece * HG + h] = make_float2(m_ref[h], lsum[h]);
                    }
                }
            }
            if (lane == 0) fence_proxy_async_smem();
            __syncwarp();
            issue_next();
            cursor_advance(cc, n, seqlens, B, max_len, NGS);
            ++it;
        }
        if (!ok) {
            // let every copy this warp started land before it leaves the shared memory
            if (lane == 0) atomicOr(status, 2u);
            for (int r = it; r < issued; ++r)
                mbar_wait_drain(&bars[warp * kRing + r % kRing], (r / kRing) & 1);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Merge for the stream kernel: one block of MW warps per (sequence, query head).
// Warp w combines pieces w, w + MW, ... (in order, eight loads in flight at a
// time); the warp results are then combined in warp order through shared memory, so the result
// does not depend on timing.
// MW warps per block: 16 when there are few streams (each with many pieces), 4 when there are
// many (each with few pieces, and the narrower blocks all fit on the GPU at once).
template <bool OUT_F32, int D, int HG, int MW>
__global__ void __launch_bounds__(MW * 32)
    decode_stream_merge_kernel(const float *__restrict__ ws_o, const float2 *__restrict__ ws_ml,
                               const int *__restrict__ seqlens, void *__restrict__ o,
                               float *__restrict__ lse, int B, int Hq, int Hkv, int max_len,
                               int nwt, unsigned *__restrict__ status)
{
    constexpr int DL = D / 32;
    constexpr int PW = 8;  // pieces per warp per round
    __shared__ float s_acc[MW][D];
    __shared__ float s_m[MW], s_l[MW];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x;
    const int b = bh / Hq, h = bh % Hq;
    const int G = Hq / Hkv, SUB = G / HG, NGS = Hkv * SUB;
    const int g = h / G, gs = (h % G) / HG, hl = (h % G) % HG;
    const int sl = g * SUB + gs;
    const long long total = warp_len_sum(seqlens, B, max_len, lane) * NGS;
    const long long base = warp_len_sum(seqlens, b, max_len, lane) * NGS;
    const long long KP = stream_slice(total, nwt);
    const int Lb = clamp_len(seqlens[b], max_len);
    const long long start = base + (long long)sl * Lb;
    const int wf = (int)(start / KP);
    int n = Lb > 0 ? (int)((start + Lb - 1) / KP) - wf + 1 : 0;
    const size_t row0 = ((size_t)wf + (size_t)b * NGS + sl) * HG + hl;  // piece j: row0 + j*HG
    if (!dbg_ok(n == 0 || row0 + (size_t)(n - 1) * HG < (size_t)nwt * HG + (size_t)B * Hq, status))
        n = 0;
    // Everything above reads only seqlens, which the stream kernel does not write: this grid is
    // launched once every stream block has passed its own dependency wait, so whatever wrote
    // seqlens before the stream kernel has finished. Only the partials need the wait, which
    // now overlaps the stream kernel's tail instead of adding a round of loads after it.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float M = -INFINITY, Ls = 0.f, acc[DL];
#pragma unroll
    for (int e = 0; e < DL; ++e) acc[e] = 0.f;
    for (int j0 = warp; j0 < n; j0 += MW * PW) {
        float2 mlj[PW];
        float x[PW][DL];
#pragma unroll
        for (int k = 0; k < PW; ++k) {
            const int j = j0 + MW * k;
            if (j < n) {
                const size_t row = row0 + (size_t)j * HG;
                mlj[k] = ws_ml[row];
                const float *src = ws_o + row * D + lane * DL;
#pragma unroll
                for (int e = 0; e < DL; ++e) x[k][e] = src[e];
            } else {
                mlj[k] = make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int e = 0; e < DL; ++e) x[k][e] = 0.f;
            }
        }
        float cm = M;
#pragma unroll
        for (int k = 0; k < PW; ++k) cm = fmaxf(cm, mlj[k].x);
        const float Mu = (cm == -INFINITY) ? 0.f : cm;
        const float a = ex2(M - Mu);
        Ls *= a;
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[e] *= a;
#pragma unroll
        for (int k = 0; k < PW; ++k) {
            const float w = ex2(mlj[k].x - Mu);
            Ls = fmaf(w, mlj[k].y, Ls);
#pragma unroll
            for (int e = 0; e < DL; ++e) acc[e] = fmaf(w, x[k][e], acc[e]);
        }
        M = cm;
    }
#pragma unroll
    for (int e = 0; e < DL; ++e) s_acc[warp][lane * DL + e] = acc[e];
    if (lane == 0) {
        s_m[warp] = M;
        s_l[warp] = Ls;
    }
    __syncthreads();
    if (warp == 0) {
        float Mt = s_m[0];
#pragma unroll
        for (int w2 = 1; w2 < MW; ++w2) Mt = fmaxf(Mt, s_m[w2]);
        const float Mu = (Mt == -INFINITY) ? 0.f : Mt;
        float Lt = 0.f, r[DL];
#pragma unroll
        for (int e = 0; e < DL; ++e) r[e] = 0.f;
#pragma unroll 4
        for (int w2 = 0; w2 < MW; ++w2) {
            const float wgt = ex2(s_m[w2] - Mu);
            Lt = fmaf(wgt, s_l[w2], Lt);
#pragma unroll
            for (int e = 0; e < DL; ++e) r[e] = fmaf(wgt, s_acc[w2][lane * DL + e], r[e]);
        }
        const float inv = (n > 0 && Lt > 0.f) ? 1.f / Lt : 0.f;
#pragma unroll
        for (int e = 0; e < DL; ++e) {
            const float v = r[e] * inv;
            if (OUT_F32)
                static_cast<float *>(o)[(size_t)bh * D + lane * DL + e] = v;
            else
                static_cast<__nv_bfloat16 *>(o)[(size_t)bh * D + lane * DL + e] = __float2bfloat16_rn(v);
        }
        if (lse != nullptr && lane == 0)
            lse[bh] = (n > 0 && Lt > 0.f) ? (Mt + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
    }
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
    if (bh >= BH) return;
    const int b = bh / Hq;
    int L = seqlens[b];
    L = L < 0 ? 0 : (L > max_len ? max_len : L);
    const int n = (L + chunk - 1) / chunk;
    // seqlens is not written by the split kernel (launched after every split block passed its
    // own dependency wait); only the chunk states need the wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

// Launch as a programmatic dependent of whatever precedes it in the stream (the kernels wait
// for it before their first global read, so only their start-up overlaps it).
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int D, int HG, typename QT>
cudaError_t launch_split_t(const DecodeArgs &a, cudaStream_t st)
{
    using P = Plan<D, HG>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_split_kernel<D, HG, QT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, P::SMEM);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set[dev] = true;
    }
    const int G = a.Hq / a.Hkv;
    dim3 grid(a.nsplit, a.Hkv * (G / HG), a.B);
    return launch_pdl(decode_split_kernel<D, HG, QT>, grid, dim3(kWarps * 32), P::SMEM, st,
                      static_cast<const QT *>(a.q), static_cast<const __nv_bfloat16 *>(a.kc),
                      static_cast<const __nv_bfloat16 *>(a.vc), a.seqlens, a.ws_o, a.ws_ml,
                      a.Hq, a.Hkv, a.max_len, a.chunk, a.nsplit, a.scale_log2, a.status,
                      wait_limit_cycles());
}

int largest_group(int G)
{
    return G % 8 == 0 ? 8 : (G % 4 == 0 ? 4 : (G % 2 == 0 ? 2 : 1));
}

template <int D, int HG, bool ROPE>
cudaError_t launch_stream_t(const DecodeArgs &a, bool out_f32, cudaStream_t st)
{
    using P = Plan<D, HG>;
    constexpr auto kern = decode_stream_kernel<D, HG, ROPE>;
    static bool attr_set[64] = {};
    static int blocks_cached[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int blocks = dev < 64 ? blocks_cached[dev] : 0;
    if (dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 P::RING + P::PBUF + P::BARS);
        if (e != cudaSuccess) return e;
        int sms = 0, occ = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWarps * 32,
                                                          P::RING + P::PBUF + P::BARS);
        if (e != cudaSuccess) return e;
        blocks = sms * (occ > 0 ? occ : 1);
        if (blocks * kWarps > kStreamMaxWarps) blocks = kStreamMaxWarps / kWarps;
        if (dev < 64) {
            blocks_cached[dev] = blocks;
            attr_set[dev] = true;
        }
    }
    if (a.max_warps > 0 && blocks * kWarps > a.max_warps) blocks = a.max_warps / kWarps;
    if (blocks < 1) return cudaErrorInvalidValue;
    // partials: one row of D per (piece, head) for the warps actually launched (at most
    // kStreamMaxWarps, which decode_workspace_bytes assumes), then one float2 per row
    float *ws_o = static_cast<float *>(a.ws);
    const size_t rows = (size_t)blocks * kWarps * HG + (size_t)a.B * a.Hq;
    float2 *ws_ml = reinterpret_cast<float2 *>(ws_o + rows * D);
    RopeIn rope = {};
    if (ROPE) {
        rope.k_new = static_cast<const __nv_bfloat16 *>(a.k_new);
        rope.v_new = static_cast<const __nv_bfloat16 *>(a.v_new);
        rope.cos_t = a.cos_t;
        rope.sin_t = a.sin_t;
        rope.kc = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.kc));
        rope.vc = static_cast<__nv_bfloat16 *>(const_cast<void *>(a.vc));
    }
    e = launch_pdl(kern, dim3(blocks), dim3(kWarps * 32), P::RING + P::PBUF + P::BARS, st,
                   static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.kc),
                   static_cast<const __nv_bfloat16 *>(a.vc), a.seqlens, ws_o, ws_ml, a.B, a.Hq,
                   a.Hkv, a.max_len, a.scale_log2, a.status, rope, wait_limit_cycles());
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    const bool many = (long long)a.B * a.Hkv * (a.Hq / a.Hkv / HG) >= 128;  // streams
    cfg.gridDim = dim3(a.B * a.Hq);
    cfg.blockDim = dim3((many ? 4 : 16) * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int nwt = blocks * kWarps;
    auto merge = out_f32 ? (many ? decode_stream_merge_kernel<true, D, HG, 4>
                                 : decode_stream_merge_kernel<true, D, HG, 16>)
                         : (many ? decode_stream_merge_kernel<false, D, HG, 4>
                                 : decode_stream_merge_kernel<false, D, HG, 16>);
    return cudaLaunchKernelEx(&cfg, merge, (const float *)ws_o, (const float2 *)ws_ml, a.seqlens,
                              a.o, a.lse, a.B, a.Hq, a.Hkv, a.max_len, nwt, a.status);
}

template <int D, bool ROPE>
cudaError_t launch_stream_d(const DecodeArgs &a, bool out_f32, cudaStream_t st)
{
    switch (largest_group(a.Hq / a.Hkv)) {
    case 8: return launch_stream_t<D, 8, ROPE>(a, out_f32, st);
    case 4: return launch_stream_t<D, 4, ROPE>(a, out_f32, st);
    case 2: return launch_stream_t<D, 2, ROPE>(a, out_f32, st);
    default: return launch_stream_t<D, 1, ROPE>(a, out_f32, st);
    }
}

template <int D, typename QT>
cudaError_t launch_split_d(const DecodeArgs &a, cudaStream_t st)
{
    switch (largest_group(a.Hq / a.Hkv)) {
    case 8: return launch_split_t<D, 8, QT>(a, st);
    case 4: return launch_split_t<D, 4, QT>(a, st);
    case 2: return launch_split_t<D, 2, QT>(a, st);
    default: return launch_split_t<D, 1, QT>(a, st);
    }
}

// RoPE of the new token and its cache store. One block per (sequence, head): blockIdx.y < Hq
// rotates query head y into q_rot (fp32, unrounded); otherwise kv head y - Hq: its key is
// rotated, rounded to bf16 and stored with its value at cache row p = seqlens[b] - 1. Thread d
// handles the pair (d, d + D/2): [x1 | x2] -> [x1 cos - x2 sin | x1 sin + x2 cos].
template <int D>
__global__ void __launch_bounds__(D / 2)
    rope_append_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k_new,
                       const __nv_bfloat16 *__restrict__ v_new, const float *__restrict__ cos_t,
                       const float *__restrict__ sin_t, __nv_bfloat16 *__restrict__ kc,
                       __nv_bfloat16 *__restrict__ vc, const int *__restrict__ seqlens,
                       float *__restrict__ q_rot, int Hq, int Hkv, int max_len)
{
    constexpr int H = D / 2;
    const int b = blockIdx.x, y = blockIdx.y, d = threadIdx.x;
    const int L = clamp_len(seqlens[b], max_len);
    const int p = L > 0 ? L - 1 : 0;
    const float c = cos_t[(size_t)p * H + d], sn = sin_t[(size_t)p * H + d];
    if (y < Hq) {
        const __nv_bfloat16 *x = q + ((size_t)b * Hq + y) * D;
        const float x1 = __bfloat162float(x[d]), x2 = __bfloat162float(x[d + H]);
        float *o = q_rot + ((size_t)b * Hq + y) * D;
        o[d] = x1 * c - x2 * sn;
        o[d + H] = x1 * sn + x2 * c;
    } else if (L > 0) {
        const int g = y - Hq;
        const __nv_bfloat16 *x = k_new + ((size_t)b * Hkv + g) * D;
        const float x1 = __bfloat162float(x[d]), x2 = __bfloat162float(x[d + H]);
        const size_t row = (((size_t)b * Hkv + g) * max_len + p) * D;
        kc[row + d] = __float2bfloat16_rn(x1 * c - x2 * sn);
        kc[row + d + H] = __float2bfloat16_rn(x1 * sn + x2 * c);
        const __nv_bfloat16 *vn = v_new + ((size_t)b * Hkv + g) * D;
        vc[row + d] = vn[d];
        vc[row + d + H] = vn[d + H];
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

bool decode_fuses_rope(int B) { return B <= kStreamMaxBatch; }

int decode_chunk_len(int B, int Hkv, int max_len)
{
    // Chunked kernel (batches above the stream kernel's limit): aim for about three blocks per
    // SM of a 152-SM GB300 at the shape's largest length; chunks of 64 to 512 keys.
    const long long target = 3LL * 152;
    int chunk = 512;
    while (chunk > 64 &&
           (long long)B * Hkv * (((long long)max_len + chunk - 1) / chunk) < target)
        chunk /= 2;
    return chunk;
}

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len)
{
    if (B <= kStreamMaxBatch) {
        const size_t HG = (size_t)largest_group(Hq / Hkv);
        const size_t rows = (size_t)kStreamMaxWarps * HG + (size_t)B * Hq;
        return rows * D * sizeof(float) + rows * sizeof(float2);
    }
    const int chunk = decode_chunk_len(B, Hkv, max_len);
    const size_t nsplit = ((size_t)max_len + chunk - 1) / chunk;
    const size_t rows = (size_t)B * Hq * nsplit;
    return rows * D * sizeof(float) + rows * sizeof(float2);
}

int decode_warps_within(int B, int Hq, int Hkv, int D, int max_len, size_t bytes)
{
    const size_t row = (size_t)D * sizeof(float) + sizeof(float2);
    if (B > kStreamMaxBatch)
        return decode_workspace_bytes(B, Hq, Hkv, D, max_len) <= bytes ? kStreamMaxWarps : 0;
    const size_t HG = (size_t)largest_group(Hq / Hkv);
    const size_t rows = bytes / row;
    const size_t fixed = (size_t)B * Hq;
    if (rows <= fixed) return 0;
    size_t warps = (rows - fixed) / HG;
    if (warps > (size_t)kStreamMaxWarps) warps = kStreamMaxWarps;
    warps -= warps % kWarps;
    return (int)warps;
}

cudaError_t launch_decode(const DecodeArgs &a0, bool out_f32, cudaStream_t st)
{
    DecodeArgs a = a0;
    if (a.B <= kStreamMaxBatch) {
        if (a.q_f32) return cudaErrorInvalidValue;  // the stream kernel takes a bf16 q
        if (a.k_new != nullptr)
            return a.D == 128 ? launch_stream_d<128, true>(a, out_f32, st)
                              : launch_stream_d<64, true>(a, out_f32, st);
        return a.D == 128 ? launch_stream_d<128, false>(a, out_f32, st)
                          : launch_stream_d<64, false>(a, out_f32, st);
    }
    if (a.k_new != nullptr) return cudaErrorInvalidValue;  // RoPE runs as its own kernel here
    a.chunk = decode_chunk_len(a.B, a.Hkv, a.max_len);
    a.nsplit = (a.max_len + a.chunk - 1) / a.chunk;
    a.ws_o = static_cast<float *>(a.ws);
    a.ws_ml = reinterpret_cast<float2 *>(a.ws_o + (size_t)a.B * a.Hq * a.nsplit * a.D);
    cudaError_t e;
    if (a.q_f32)
        e = (a.D == 128) ? launch_split_d<128, float>(a, st) : launch_split_d<64, float>(a, st);
    else
        e = (a.D == 128) ? launch_split_d<128, __nv_bfloat16>(a, st)
                         : launch_split_d<64, __nv_bfloat16>(a, st);
    if (e != cudaSuccess) return e;
    if (a.D == 128)
        e = out_f32 ? launch_merge<true, 128>(a, st) : launch_merge<false, 128>(a, st);
    else
        e = out_f32 ? launch_merge<true, 64>(a, st) : launch_merge<false, 64>(a, st);
    return e;
}

cudaError_t launch_rope_append(const void *q, const void *k_new, const void *v_new,
                               const float *cos_t, const float *sin_t, void *kc, void *vc,
                               const int *seqlens, float *q_rot, int B, int Hq, int Hkv, int D,
                               int max_len, cudaStream_t st)
{
    dim3 grid(B, Hq + Hkv);
    if (D == 128)
        rope_append_kernel<128><<<grid, 64, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k_new),
            static_cast<const __nv_bfloat16 *>(v_new), cos_t, sin_t,
            static_cast<__nv_bfloat16 *>(kc), static_cast<__nv_bfloat16 *>(vc), seqlens, q_rot,
            Hq, Hkv, max_len);
    else
        rope_append_kernel<64><<<grid, 32, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k_new),
            static_cast<const __nv_bfloat16 *>(v_new), cos_t, sin_t,
            static_cast<__nv_bfloat16 *>(kc), static_cast<__nv_bfloat16 *>(vc), seqlens, q_rot,
            Hq, Hkv, max_len);
    return cudaGetLastError();
}

}  // namespace gqa
