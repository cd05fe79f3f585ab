// prefill_tc.cu -- fused attention forward (prefill) on sm_103a tensor cores, bf16 in,
// fp32 accumulation and softmax state, head dim 128 or 64. q, k, v are read through 4-D tensor
// maps, so any layout with a contiguous head dim and 16-byte multiple strides works in place
// (the [B, H, S, D] default, [B, S, H, D], or q/k/v as slices of one fused projection output).
//
// One thread block owns 256 consecutive query rows of one (batch, query head): two 128-row
// Q tiles (HD = 128; half as wide at 64). Both tiles consume the same stream of 128-key K/V
// tiles, so every K/V tile brought in by TMA feeds four tensor-core products. Roles (12 warps,
// three warpgroups; the first gives registers to the other two at entry):
//   warp 0      TMA producer: Q tiles once, then K_j into a 2-stage and V_j into a 3-stage ring
//               (V also waits for its conversion, so it gets one stage more);
//   warp 1      tcgen05 issuer (the warp runs converged, one elected lane issues each MMA):
//               S_t = Q_t K_j^T into TMEM, O_t += P_t V_j with P_t read from TMEM; owns the
//               TMEM allocation;
//   warps 2-3   convert each landed V tile from bf16 to fp16 in place (see below), unless
//               V was converted beforehand;
//   warps 4-7   softmax for tile 0, warps 8-11 for tile 1:
//               one thread per query row (its TMEM lane). Reads the 128 scores of its row,
//               masks, updates the running max and sum, writes P (fp16) over the scores it
//               came from, rescales its O row when the max moved, and finally writes O / l
//               and the LSE.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1, 128 fp32 columns each (O uses HD of them); P_t is
// packed fp16 in the first 64 columns of S_t. S and P never leave the SM.
//
// Precision of the P V product: P is rounded to a 16-bit type before the tensor core consumes
// it. With bf16 (8-bit significand) a peaky softmax (a few keys carrying most of the weight)
// showed errors near 8e-3 in the output; fp16 (11-bit significand) brings that to about 1e-3.
// The tensor core needs both operands of one product in the same type, so V is converted to
// fp16. fp16 spans only 2^-14 .. 65504 with full precision, so every (batch, kv head) slab of V
// gets a power-of-two scale 2^-e chosen from its largest finite |v|: e = 0 while that maximum
// lies in [2^-9, 2^16) (every bf16 value there converts exactly, or with an error far below the
// output's rounding), otherwise e puts the maximum in [2^14, 2^15), which keeps every value
// within 2^28 of the maximum exact. O is linear in V, so the epilogue multiplies by 2^e and the
// result is the same as with unscaled V, for any finite bf16 V. Normally a separate HBM-bound
// kernel (convert_v_kernel) writes an fp16 copy of V once per call, with e = 0, and records each
// block's maximum per slab; v_scale_kernel (one block per slab) picks e and rewrites the rare
// slabs that need e != 0; the attention kernel streams the copy and reads e only for its
// epilogue. Every V tile is read by many blocks (all heads of its group, all later row blocks),
// and converting it in shared memory in each of them cost more than the copy; the conversion
// also competed with the scores MMAs for shared-memory bandwidth (the tensor core wins), which
// made it the slowest stage of the pipeline. When no scratch is available for the copy (stream
// capture before the scratch has grown that far; a copy above 1 GiB) warps 2-3 convert each
// landed tile in place instead, with the slab's scale from the same two small kernels; both ways
// give the same fp16 values.
//
// The two tiles alternate on the tensor core: while tile 0's softmax runs, the tensor core
// computes tile 1's P V and next S, and the other way round. Issue order per key tile j:
//   [PV_0(j-1)] S_0(j) [PV_1(j-1)] S_1(j)
// tcgen05 operations of one thread complete in issue order, so the commit that signals
// "S_t(j) ready" also guarantees PV_t(j-1) finished: the softmax may then overwrite P_t and
// rescale O_t without a separate barrier.
//
// Rescaling is lazy: a row keeps its reference max until the true max exceeds it by more than
// 2^8 (scores are in log2 units), so the O row in TMEM is rescaled only then. The result is
// the same in exact arithmetic because the same reference is used for O and l.
//
// Sources: "Attention three-op fusion" (xdnf.cn/news/349386): section 1.1 and 1.2 (S = QK^T
// scale, softmax, O = PV; S and P must stay on chip), section 2.2-2.3 (running max and sum,
// correction factor exp(m - m_new) applied to the accumulated output, one division by l at the
// end), section 3.3 and 5.5 (m, l and the accumulator in fp32), section 4.3 (causal mask: key
// tiles above the diagonal are skipped, the diagonal tile is masked per element with -inf),
// section 6.1 (ragged tail: out-of-range K/V rows read as 0, their scores set to -inf);
// "triton-optimization" skill (skillsmp.com) section 3.5 (LSE = m + log l).
#include "internal.h"
#include "ptx.cuh"

#include <algorithm>
#include <array>
#include <cmath>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

namespace gqa {
namespace {

constexpr int BM = 128;        // query rows per tile = TMEM lanes
constexpr int BN = 128;        // keys per K/V tile
constexpr int kThreads = 384;  // 12 warps = 3 warpgroups
// Registers per thread: the block is compiled for (and launched with) kRegsLaunch; at entry the
// producer / issuer / converter warpgroup gives registers back (kRegsLow) and the two softmax
// warpgroups, which hold a row of 128 scores per thread, take them (kRegsHigh). Each SMSP holds
// one warp of each warpgroup. An increase that the block's pool cannot cover would wait
// forever, so the host checks the compiled count before the first launch.
constexpr int kRegsLaunch = 168, kRegsLow = 136, kRegsHigh = 184;
static_assert(kRegsLow * 128 + kRegsHigh * 256 <= kRegsLaunch * kThreads, "register pool");
constexpr uint32_t kBox = 16384;          // one 128-row x 64-col bf16 box (128-byte rows)
constexpr int KST = 2;                    // K ring stages
constexpr int VST = 3;                    // V ring stages (V also waits for its fp16 conversion)
// K_jj reuses K_jj-2's stage (read by the scores of step jj - 2) and V_jj reuses V_jj-3's (read by
// the P V of step jj - 2): one "step jj - 2 done" barrier covers both.
static_assert(KST == 2 && VST == 3, "stage reuse tied to step jj - 2");
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// Shared-memory plan for head dim HD (64 or 128): two Q tiles, the K ring, the V ring, then the
// barriers. A tile is 128 rows x HD bf16, stored as HD / 64 boxes of 64 columns.
template <int HD>
struct Geo {
    static_assert(HD == 64 || HD == 128, "head dim");
    static constexpr int NBOX = HD / 64;
    static constexpr uint32_t kTile = NBOX * kBox;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = 2 * kTile;
    static constexpr uint32_t kOffV = kOffK + KST * kTile;
    static constexpr uint32_t kOffBar = kOffV + VST * kTile;
    static constexpr uint32_t kSmem = kOffBar + 256 + 1024;  // + barriers, + alignment slack
    static_assert(kSmem <= 232448, "shared memory per block");
};

// TMEM column bases
constexpr uint32_t kColS = 0;    // + 128 t
constexpr uint32_t kColO = 256;  // + 128 t

// barrier indices
enum : int {
    B_Q = 0,
    B_KFULL = 1,                // KST
    B_STEP = B_KFULL + KST,     // 2: all MMAs of key step jj done (by parity of jj); the K and
                                // V stages that step n reuses are both freed by step n - 2
    B_VFULL = B_STEP + 2,       // VST
    B_VREADY = B_VFULL + VST,   // VST: V stage converted to fp16
    B_SFULL = B_VREADY + VST,   // 2 (per tile)
    B_PFULL = B_SFULL + 2,      // 2 (per tile)
    B_OFULL = B_PFULL + 2,      // 2 (per tile)
    B_DRAIN = B_OFULL + 2,
    B_ML = B_DRAIN + 1,         // pair mode: both softmax warpgroups posted their (m, l)
    NUM_BARS = B_ML + 1
};
static_assert(NUM_BARS * 8 + 8 <= 256, "barrier area");

__host__ __device__ __forceinline__ int last_key_tile(int causal, int q_first, int nkv)
{
    // causal: the tile whose rows start at key position q_first needs keys up to q_first + 127
    // (-1: no key at all)
    if (!causal) return nkv - 1;
    const int last = q_first + BM - 1;
    if (last < 0) return -1;
    const int lim = last / BN;
    return lim < nkv - 1 ? lim : nkv - 1;
}

// Key tiles that the row block rb of `rows` rows (256, or 128 in pair mode) visits: every tile
// up to the one holding its last row (causal), or all of them.
__host__ __device__ __forceinline__ int rb_key_tiles(int rb, int S, int causal, int rows)
{
    const int nkv = (S + BN - 1) / BN;
    if (!causal) return nkv;
    const int q0 = rb * rows;
    const int qlast = (q0 + rows < S ? q0 + rows : S) - 1;
    const int l = qlast / BN;
    return (l < nkv - 1 ? l : nkv - 1) + 1;
}

// Split mode: row block rb is cut into ceil(tiles / J) segments of at most J key tiles, each
// one block. Every row block gets the same number of segment slots, NS (the longest row
// block's segment count), so block -> (row block, segment, head) is plain arithmetic: blocks
// are numbered heaviest row block first (row block n_rb - 1 - blockIdx / (NS * heads)), then
// segment, then batch x head. Slots past a row block's segments exit at once.
__host__ __device__ __forceinline__ int rb_segments(int rb, int S, int causal, int J, int rows)
{
    return (rb_key_tiles(rb, S, causal, rows) + J - 1) / J;
}

// Segment slots per row block in split mode: the most segments any row block has.
__host__ __device__ __forceinline__ int split_slots(int S, int causal, int J, int rows)
{
    const int n_rb = (S + rows - 1) / rows;
    const int a = rb_segments(n_rb - 1, S, causal, J, rows), b = rb_segments(0, S, causal, J, rows);
    return a > b ? a : b;
}

// Largest finite magnitude among the bf16 halves of the four words of c, folded into `acc` as
// two 16-bit lanes of magnitude bits (inf and NaN count as 0: no scale can bring them into the
// fp16 range, and they propagate as they would in fp32).
__device__ __forceinline__ uint32_t absmax_acc(uint32_t acc, uint4 c)
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t a = w[e] & 0x7FFF7FFFu;
        acc = __vmaxu2(acc, a & __vcmpltu2(a, 0x7F807F80u));
    }
    return acc;
}

// Exponent e of a V slab's scale from its largest finite |v| (bf16 magnitude bits m): 0 while
// the maximum lies in [2^-9, 2^16), else the e that puts it in [2^14, 2^15), within [-126, 113]
// so that 2^e and 2^-e are normal fp32 numbers.
__host__ __device__ __forceinline__ int v_scale_exponent(uint32_t m)
{
    if (m == 0) return 0;
    int E;
    if (m >= 0x80u) {
        E = (int)((m >> 7) & 0xFFu) - 127;
    } else {  // bf16 subnormal: m * 2^-133
        int top = 0;
        while ((m >> (top + 1)) != 0) ++top;
        E = top - 133;
    }
    if (E >= -9 && E <= 15) return 0;
    const int e = E - 14;
    return e < -126 ? -126 : e;
}

// 2^e as an fp32 number, e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// Two bf16 (one 32-bit word) -> two fp16 of (value * s), round to nearest even. s is a power of
// two that keeps every finite value of the slab within the fp16 range, so nothing saturates.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float s)
{
    return pack_f16x2(bf16lo(w) * s, bf16hi(w) * s);
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    return pack_f16x2(bf16lo(w), bf16hi(w));
}

// Zeroes rows >= rows_ok of a 128-row bf16 tile of nchunk 16-byte chunks (64-column boxes of
// 1024 chunks, 8 per row): the chunks ct, ct + 64, ... only.
// Out of line on purpose: inlined (or folded into the conversion loop as a per-chunk select) it
// cost the whole kernel 2-12% on full-length prefill, where it never runs.
__device__ __noinline__ void zero_v_tail(uint4 *tile, int ct, int rows_ok, int nchunk)
{
    for (int c = ct; c < nchunk; c += 64)
        if (((c & 1023) >> 3) >= rows_ok) tile[c] = make_uint4(0, 0, 0, 0);
}

// HD: head dim (64 or 128). The tensor maps are 4-D {HD, rows, heads, batch} with any strides,
// so q, k and v may be views (a [B, S, H, D] layout, a fused QKV projection output); O is
// written at out + b o_sb + i o_ss + h o_sh (elements), the LSE as [B, Hq, S].
// SPLIT = false: one block per (row block, head, batch), final O and LSE.
// SPLIT = true: one block per (row block, key segment of J tiles, head, batch); it writes the
// segment's normalised O (fp32) and its LSE (log2 units) to ws_o / ws_lse, and
// prefill_split_merge_kernel combines the segments of each row.
// VPRE = true: tv maps an fp16 copy of V written by convert_v_kernel (warps 2-3 have nothing to
// do). VPRE = false: tv maps the bf16 V, converted on chip by warps 2-3.
// vexp[b * Hkv + g]: the exponent e of V slab (b, g)'s scale (V is used as v * 2^-e, so O is
// multiplied by 2^e), written by convert_v_kernel, which this grid depends on (programmatic
// dependent launch): every thread that reads it first waits for that grid.
template <int HD, bool OUT_F32, bool SPLIT, bool VPRE, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, void *__restrict__ out,
                      float *__restrict__ lse, int B, int S, int Hq, int Hkv, float scale_log2,
                      int causal, unsigned *__restrict__ status, int J, float *__restrict__ ws_o,
                      float *__restrict__ ws_lse, const int *__restrict__ kv_lens, int max_kv,
                      int front, long long o_sb, long long o_ss, long long o_sh, int NS,
                      const int *__restrict__ vexp, long long wait_limit)
{
    using G = Geo<HD>;
    constexpr uint32_t kTile = G::kTile, kOffQ = G::kOffQ, kOffK = G::kOffK, kOffV = G::kOffV,
                       kOffBar = G::kOffBar;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr int kSoftmaxWarp0 = 4;  // first of the 8 softmax warps

    // ---- work item: heaviest row blocks first (causal), heads of one group adjacent
    constexpr int RB = PAIR ? BM : 2 * BM;  // query rows per block
    const int n_rb = (S + RB - 1) / RB;
    int rb, hb, seg = 0;
    if (!SPLIT) {
        rb = n_rb - 1 - (int)blockIdx.x / (Hq * B);
        hb = (int)blockIdx.x % (Hq * B);
    } else {
        const int per_rb = NS * Hq * B;
        rb = n_rb - 1 - (int)blockIdx.x / per_rb;
        const int rem = (int)blockIdx.x % per_rb;
        seg = rem / (Hq * B);
        hb = rem % (Hq * B);
        if (seg >= rb_segments(rb, S, causal, J, RB)) return;  // empty slot: nothing set up yet
    }
    const int h = hb % Hq, b = hb / Hq;
    const int g = h / (Hq / Hkv);
    const int q0 = rb * RB;
    // the block's work item must lie inside the problem (nothing is set up yet: leave at once)
    if (!dbg_ok(rb >= 0 && rb < n_rb && b < B && g < Hkv, status)) return;
    // Keys: L of them. Plain prefill: L = S. Chunk against a cache (kv_lens given): the S
    // queries are the last S of the L_b cached tokens, so query row i sits at key position
    // i + off, off = L_b - S.
    int L = S;
    if (kv_lens != nullptr) {
        L = kv_lens[b];
        if (L < 0 || L > max_kv) {
            if (threadIdx.x == 0 && rb == n_rb - 1 && h == 0) atomicOr(status, 1u);
            L = L < 0 ? 0 : max_kv;
        }
    }
    // front != 0 (padded batch): the L valid queries are rows 0..L-1 (off = 0) and rows >= L
    // are padding that sees no key
    const int off = front ? 0 : L - S;
    const int nkv = (L + BN - 1) / BN;
    // Q tiles loaded: two (rows q0.., q0 + 128..), or one in pair mode, where both softmax
    // warpgroups work on the same 128 rows and take the block's key tiles in turns
    const int n_tiles = (!PAIR && q0 + BM < S) ? 2 : 1;
    int last_j[2];
    last_j[0] = (front && q0 >= L) ? -1 : last_key_tile(causal, q0 + off, nkv);
    last_j[1] = (!PAIR && n_tiles == 2 && !(front && q0 + BM >= L))
                    ? last_key_tile(causal, q0 + BM + off, nkv)
                    : -1;
    const int n_j = max(last_j[0], last_j[1]) + 1;  // 0: no key at all (O = 0, LSE = -inf)
    // key tiles [jb, je) of this block. Tile t (softmax warpgroup t) works on the tiles from
    // first_j[t] to hi[t], every tile (two Q tiles) or every other one (pair mode: tile t takes
    // jb + t, jb + t + 2, ...); it has none when hi[t] < first_j[t].
    const int jb = SPLIT ? seg * J : 0;
    const int je = SPLIT ? min(jb + J, n_j) : n_j;
    const int nJ = je - jb;
    int hi[2], first_j[2];
    if (PAIR) {
        for (int t = 0; t < 2; ++t) {
            first_j[t] = jb + t;
            const int last = je - 1;
            hi[t] = (((last - jb) & 1) == t) ? last : last - 1;
        }
    } else {
        first_j[0] = first_j[1] = jb;
        hi[0] = min(je - 1, last_j[0]);
        hi[1] = min(je - 1, last_j[1]);
    }

    if (!SPLIT && n_j == 0) {
        // No row of the block sees a key (padding rows of a padded batch, an empty sequence):
        // O = 0 and LSE = -inf, written without setting up barriers, TMEM or the roles.
        for (int idx = threadIdx.x; idx < RB * (HD / 8); idx += kThreads) {
            const int i = q0 + idx / (HD / 8), c = idx % (HD / 8);
            if (i >= S) continue;
            const long long e = b * o_sb + h * o_sh + (long long)i * o_ss + c * 8;
            if (OUT_F32) {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + e);
                dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) + e) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (lse != nullptr)
            for (int r = threadIdx.x; r < RB; r += kThreads)
                if (q0 + r < S) lse[((size_t)b * Hq + h) * S + q0 + r] = -INFINITY;
        return;
    }

    if (threadIdx.x == 0) {
        mbar_init(&bar[B_Q], 1);
        for (int s = 0; s < KST; ++s) mbar_init(&bar[B_KFULL + s], 1);
        for (int s = 0; s < 2; ++s) mbar_init(&bar[B_STEP + s], 1);
        for (int s = 0; s < VST; ++s) {
            mbar_init(&bar[B_VFULL + s], 1);
            mbar_init(&bar[B_VREADY + s], 64);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar[B_SFULL + t], 1);
            mbar_init(&bar[B_PFULL + t], BM);
            mbar_init(&bar[B_OFULL + t], 1);
        }
        mbar_init(&bar[B_DRAIN], 1);
        mbar_init(&bar[B_ML], 2 * BM);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
        // ================================================================ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tq);
            tma_prefetch_desc(&tk);
            tma_prefetch_desc(&tv);
            mbar_arrive_expect_tx(&bar[B_Q], n_tiles * kTile);
            for (int t = 0; t < n_tiles; ++t)
                for (int x = 0; x < G::NBOX; ++x)
                    tma_load_4d(smem + kOffQ + t * kTile + x * kBox, &tq, &bar[B_Q], x * 64,
                                q0 + t * BM, h, b);
            int issued_k[KST] = {}, issued_v[VST] = {};
            auto load_k = [&](int jj) {
                const int sk = jj % KST, uk = jj / KST;
                mbar_arrive_expect_tx(&bar[B_KFULL + sk], kTile);
                for (int x = 0; x < G::NBOX; ++x)
                    tma_load_4d(smem + kOffK + sk * kTile + x * kBox, &tk, &bar[B_KFULL + sk],
                                x * 64, (jb + jj) * BN, g, b);
                issued_k[sk] = uk + 1;
            };
            // the first KST key tiles need no stage to be freed: load them before waiting for
            // the V conversion, so the first scores of both tiles can run meanwhile
            for (int jj = 0; jj < KST && jj < nJ; ++jj) load_k(jj);
            for (int jj = 0; jj < nJ; ++jj) {
                const int j = jb + jj;
                // K_jj and V_jj reuse the stages of K_jj-2 and V_jj-3, both last read by the
                // MMAs of step jj - 2
                if (jj >= 2 &&
                    !mbar_wait(&bar[B_STEP + ((jj - 2) & 1)], ((jj - 2) >> 1) & 1, abort_flag, wait_limit))
                    break;
                if (jj >= KST) load_k(jj);
                // the fp16 copy of V comes from the conversion kernel just before this one,
                // which lets this grid start early (programmatic dependent launch): everything
                // up to here overlaps its tail
                if (VPRE && jj == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
                const int sv = jj % VST, uv = jj / VST;
                mbar_arrive_expect_tx(&bar[B_VFULL + sv], kTile);
                for (int x = 0; x < G::NBOX; ++x)
                    tma_load_4d(smem + kOffV + sv * kTile + x * kBox, &tv, &bar[B_VFULL + sv],
                                x * 64, j * BN, g, b);
                issued_v[sv] = uv + 1;
            }
            // Every load of this block is issued: warm L2 with the Q tiles of the block that
            // will most likely run on this SM next (one block per SM at a time, launched in
            // order, so about one SM count further on), whose set-up otherwise waits on DRAM.
            if (!SPLIT) {
                uint32_t nsm;
                asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
                const int nb = (int)blockIdx.x + (int)nsm;
                if (nb < (int)gridDim.x) {
                    const int nrb = n_rb - 1 - nb / (Hq * B), nhb = nb % (Hq * B);
                    const int nq0 = nrb * RB;
                    for (int t = 0; t < (PAIR ? 1 : 2) && nq0 + t * BM < S; ++t)
                        for (int x = 0; x < G::NBOX; ++x)
                            tma_prefetch_4d(&tq, x * 64, nq0 + t * BM, nhb % Hq, nhb / Hq);
                }
            }
            if (*abort_flag) {
                // let every copy this block started land before the block exits
                mbar_wait_drain(&bar[B_Q], 0);
                for (int s = 0; s < KST; ++s)
                    if (issued_k[s]) mbar_wait_drain(&bar[B_KFULL + s], (issued_k[s] - 1) & 1);
                for (int s = 0; s < VST; ++s)
                    if (issued_v[s]) mbar_wait_drain(&bar[B_VFULL + s], (issued_v[s] - 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ================================================================ tcgen05 issuer
        // The whole warp runs this loop converged; one elected lane issues each MMA and commit.
        constexpr unsigned FULL = 0xffffffffu;
        constexpr uint32_t idS = idesc_f32acc(BM, BN, 0, 0, 1);  // bf16 Q, K: K-major
        constexpr uint32_t idO = idesc_f32acc(BM, HD, 0, 1, 0);  // fp16 P (TMEM), V MN-major
        const uint32_t sQ = smem_u32(smem + kOffQ);
        const uint32_t sK = smem_u32(smem + kOffK);
        const uint32_t sV = smem_u32(smem + kOffV);
        // O_t += P_t V_(jj-1): the P V of key tile jb + jj - 1 for tile t, its kp-th P
        auto issue_pv = [&](int t, int jj, int kp) {
            const uint32_t vbase = sV + ((jj - 1) % VST) * kTile;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                // B = V rows 16kk..16kk+15: MN-major, 64-col chunks 16 KB apart (one chunk when
                // HD = 64), 8-row groups 1 KB apart
                const uint64_t bd = smem_desc_sw128(vbase + kk * 2048, kBox, 1024);
                mma_ts_warp(tmem + kColO + t * 128, tmem + kColS + t * 128 + kk * 8, bd, idO,
                            (kp > 0 || kk > 0) ? 1u : 0u);
            }
            if (jb + jj - 1 == hi[t]) mma_commit_warp(&bar[B_OFULL + t]);
        };
        // S_t = Q K_jj^T (Q tile t, or the block's one Q tile in pair mode)
        auto issue_s = [&](int t, int jj) {
            const uint32_t qbase = sQ + (PAIR ? 0 : t) * kTile;
            const uint32_t kbase = sK + (jj % KST) * kTile;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                const uint64_t ad = smem_desc_sw128(qbase + off, 16, 1024);
                const uint64_t bd = smem_desc_sw128(kbase + off, 16, 1024);
                mma_ss_warp(tmem + kColS + t * 128, ad, bd, idS, kk > 0 ? 1u : 0u);
            }
            mma_commit_warp(&bar[B_SFULL + t]);
        };
        bool ok = __all_sync(FULL, mbar_wait(&bar[B_Q], 0, abort_flag, wait_limit));
        for (int jj = 0; ok && jj <= nJ; ++jj) {
            const int j = jb + jj;
            const bool do_s = jj < nJ;
            const bool do_pv = jj >= 1;
            if (do_s &&
                !__all_sync(FULL, mbar_wait(&bar[B_KFULL + jj % KST], (jj / KST) & 1, abort_flag, wait_limit)))
                break;
            const int vbar = (VPRE ? B_VFULL : B_VREADY) + (jj - 1) % VST;  // V_jj-1 usable
            if constexpr (PAIR) {
                // Key tile j belongs to tile (j - jb) & 1. The scores go first: their tile's
                // previous P was read by a P V issued in an earlier step (tcgen05 operations
                // complete in order), so they need no P, and the other tile's softmax is not
                // held up by this one's.
                const int ts = jj & 1, tp = (jj - 1) & 1;
                tc_fence_after();
                if (do_s && j <= hi[ts]) issue_s(ts, jj);
                if (do_pv && j - 1 <= hi[tp]) {
                    const int kp = (jj - 1) >> 1;  // tile tp's P number
                    if (!__all_sync(FULL, mbar_wait(&bar[vbar], ((jj - 1) / VST) & 1, abort_flag, wait_limit)) ||
                        !__all_sync(FULL, mbar_wait(&bar[B_PFULL + tp], kp & 1, abort_flag, wait_limit)))
                        break;
                    tc_fence_after();
                    issue_pv(tp, jj, kp);
                }
            } else {
                if (do_pv &&
                    !__all_sync(FULL, mbar_wait(&bar[vbar], ((jj - 1) / VST) & 1, abort_flag, wait_limit)))
                    break;
                tc_fence_after();
                for (int t = 0; t < 2 && ok; ++t) {
                    if (do_pv && j - 1 <= hi[t]) {
                        if (!__all_sync(FULL, mbar_wait(&bar[B_PFULL + t], (jj - 1) & 1, abort_flag, wait_limit))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(t, jj, jj - 1);
                    }
                    if (do_s && j <= hi[t]) issue_s(t, jj);
                }
                if (!ok) break;
            }
            mma_commit_warp(&bar[B_STEP + (jj & 1)]);  // frees K_jj and V_jj-1
        }
        // drain: all issued tcgen05 work finishes before TMEM is released
        mma_commit_warp(&bar[B_DRAIN]);
        mbar_wait_drain(&bar[B_DRAIN], 0);
        __syncwarp();
    } else if (!VPRE && (warp == 2 || warp == 3)) {
        // ================================================================ V bf16 -> fp16
        // The P V product runs in fp16 (10-bit mantissa for P instead of bf16's 7): each V tile
        // is converted in place, with the slab's scale, once it lands, then handed to the tensor
        // core.
        const int ct = threadIdx.x - 64;
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const float vsc = exp2i(-vexp[b * Hkv + g]);  // this slab's scale 2^-e
        for (int jj = 0; jj < nJ; ++jj) {
            const int s = jj % VST;
            if (!__all_sync(0xffffffffu, mbar_wait(&bar[B_VFULL + s], (jj / VST) & 1, abort_flag, wait_limit)))
                break;
            uint4 *tile = reinterpret_cast<uint4 *>(smem + kOffV + s * kTile);
            // rows at or past L (a cache's stale rows may hold anything) become 0 first: p is
            // 0 there, but 0 * NaN would not be. Each thread zeroes only the chunks it converts
            // below, so program order is the only ordering needed.
            const int rows_ok = L - (jb + jj) * BN;  // >= BN except on the tile holding L
            if (rows_ok < BN) zero_v_tail(tile, ct, rows_ok, (int)(kTile / 16));
#pragma unroll 4
            for (int c = ct; c < (int)(kTile / 16); c += 64) {
                uint4 w = tile[c];
                w.x = bf16x2_to_f16x2_scaled(w.x, vsc);
                w.y = bf16x2_to_f16x2_scaled(w.y, vsc);
                w.z = bf16x2_to_f16x2_scaled(w.z, vsc);
                w.w = bf16x2_to_f16x2_scaled(w.w, vsc);
                tile[c] = w;
            }
            fence_proxy_async_smem();
            mbar_arrive(&bar[B_VREADY + s]);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ================================================================ softmax / epilogue
        const int t = (warp - kSoftmaxWarp0) / 4;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // row within the tile = TMEM lane
        const int i = q0 + (PAIR ? 0 : t) * BM + r;  // query row
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t tS = lane_base + kColS + t * 128;
        const uint32_t tO = lane_base + kColO + t * 128;
        if (PAIR || t < n_tiles) {
            float m_ref = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = first_j[t]; j <= hi[t]; j += PAIR ? 2 : 1) {
                const int jj = PAIR ? (j - first_j[t]) >> 1 : j - jb;  // this tile's step number
                ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_SFULL + t], jj & 1, abort_flag, wait_limit));
                if (!ok) break;
                tc_fence_after();
                uint32_t sv[128];  // raw fp32 bits of the row's scores
                tmem_ld128(tS, sv);
                const int k0 = j * BN;
                const bool dead = front && i >= L;  // padding row
                if (k0 + BN > L || (causal && k0 + BN - 1 > i + off) || dead) {
                    const int lim = dead ? 0 : (causal ? min(i + off + 1, L) : L);  // keys < lim
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (k0 + c >= lim) sv[c] = __float_as_uint(-INFINITY);
                }
                // row max: four independent chains of three-input max
                float mc[4];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float a = __uint_as_float(sv[32 * q4]);
#pragma unroll
                    for (int e = 1; e < 31; e += 2)
                        a = fmax3(a, __uint_as_float(sv[32 * q4 + e]),
                                  __uint_as_float(sv[32 * q4 + e + 1]));
                    mc[q4] = fmaxf(a, __uint_as_float(sv[32 * q4 + 31]));
                }
                const float mx = fmax3(mc[0], mc[1], fmaxf(mc[2], mc[3]));
                const float m_cand = mx * scale_log2;
                const bool need = m_cand > m_ref + kRescaleThreshold;
                const float m_new = need ? m_cand : m_ref;
                const float mu = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = ex2(m_ref - mu);
                const float2 sc2 = make_float2(scale_log2, scale_log2);
                const float2 nm2 = make_float2(-mu, -mu);
                float2 rsa = make_float2(0.f, 0.f), rsb = rsa;
#pragma unroll
                for (int half = 0; half < 2; ++half) {  // 32 packed columns at a time
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int e = half * 64 + 2 * c;
                        const float2 x = ffma2(make_float2(__uint_as_float(sv[e]),
                                                           __uint_as_float(sv[e + 1])),
                                               sc2, nm2);
                        const float2 p = make_float2(ex2(x.x), ex2(x.y));
                        if (c & 1)
                            rsb = fadd2(rsb, p);
                        else
                            rsa = fadd2(rsa, p);
                        pk[c] = pack_f16x2(p.x, p.y);
                    }
                    tmem_st32(tS + half * 32, pk);
                }
                l = fmaf(l, alpha, (rsa.x + rsa.y) + (rsb.x + rsb.y));
                if (jj > 0 && __any_sync(0xffffffffu, need)) {
                    uint32_t ov[HD];
                    if constexpr (HD == 128) {
                        tmem_ld128(tO, ov);
                    } else {
                        tmem_ld32(tO, ov);
                        tmem_ld32(tO + 32, ov + 32);
                    }
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int e = 0; e < HD / 2; ++e) {
                        const float2 v2 = fmul2(make_float2(__uint_as_float(ov[2 * e]),
                                                            __uint_as_float(ov[2 * e + 1])),
                                                a2);
                        ov[2 * e] = __float_as_uint(v2.x);
                        ov[2 * e + 1] = __float_as_uint(v2.y);
                    }
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) tmem_st32(tO + c * 32, &ov[c * 32]);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bar[B_PFULL + t]);
                m_ref = m_new;
            }
            const bool active = hi[t] >= first_j[t];  // warp-uniform
            // V was used as v * 2^-e: O comes out multiplied by 2^e. The exponent is read
            // before the wait for the last P V, so its latency overlaps that wait.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            const int vexp_e = vexp[b * Hkv + g];
            if (ok && active)
                ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_OFULL + t], 0, abort_flag, wait_limit));
            // a row block whose keys fit in one segment writes its final result directly
            const bool direct = SPLIT && rb_segments(rb, S, causal, J, RB) == 1;
            const float osc = exp2i(vexp_e);
            if constexpr (PAIR) {
                // Both warpgroups hold (m, l, O) of the same rows over different key tiles. Each
                // posts its (m, l) in the second Q buffer (never loaded in pair mode), then
                // combines its half of the columns of both O accumulators with the weights
                // 2^(m_t - M) and writes them (an empty segment or a row that sees no key: O = 0,
                // LSE = -inf).
                constexpr unsigned FULL = 0xffffffffu;
                float *ml = reinterpret_cast<float *>(smem + kOffQ + kTile);
                ml[(t * BM + r) * 2] = active ? m_ref : -INFINITY;
                ml[(t * BM + r) * 2 + 1] = active ? l : 0.f;
                mbar_arrive(&bar[B_ML]);
                if (ok) ok = __all_sync(FULL, mbar_wait(&bar[B_ML], 0, abort_flag, wait_limit));
                const int u = 1 - t;
                const bool active_u = hi[u] >= first_j[u];
                if (ok && active_u)
                    ok = __all_sync(FULL, mbar_wait(&bar[B_OFULL + u], 0, abort_flag, wait_limit));
                if (ok) {
                    tc_fence_after();
                    const float mt = active ? m_ref : -INFINITY, lt = active ? l : 0.f;
                    const float mu = ml[(u * BM + r) * 2], lu = ml[(u * BM + r) * 2 + 1];
                    const float M = fmaxf(mt, mu);
                    const float Mz = (M == -INFINITY) ? 0.f : M;
                    const float wt = active ? ex2(mt - Mz) : 0.f;
                    const float wu = active_u ? ex2(mu - Mz) : 0.f;
                    const float Ls = wt * lt + wu * lu;
                    const float inv = Ls > 0.f ? osc / Ls : 0.f;
                    const float ct = wt * inv, cu = wu * inv;
                    const bool part = SPLIT && !direct;
                    const bool live = i < S;
                    const uint32_t tOu = lane_base + kColO + u * 128;
                    const size_t prow = (size_t)blockIdx.x * RB + r;
                    const long long obase = b * o_sb + h * o_sh + (long long)(live ? i : 0) * o_ss;
#pragma unroll 1
                    for (int c = t * (HD / 64); c < (t + 1) * (HD / 64); ++c) {
                        uint32_t a[32], bu[32];
                        if (active)
                            tmem_ld32(tO + c * 32, a);
                        else
#pragma unroll
                            for (int e = 0; e < 32; ++e) a[e] = 0u;
                        if (active_u)
                            tmem_ld32(tOu + c * 32, bu);
                        else
#pragma unroll
                            for (int e = 0; e < 32; ++e) bu[e] = 0u;
                        if (!live) continue;
                        float x[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            x[e] = fmaf(ct, __uint_as_float(a[e]), cu * __uint_as_float(bu[e]));
                        if (part || OUT_F32) {
                            float4 *dst = reinterpret_cast<float4 *>(
                                part ? ws_o + prow * HD + c * 32
                                     : static_cast<float *>(out) + obase + c * 32);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                dst[e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(
                                static_cast<__nv_bfloat16 *>(out) + obase + c * 32);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                dst[e] = make_uint4(pack_bf16x2(x[8 * e], x[8 * e + 1]),
                                                    pack_bf16x2(x[8 * e + 2], x[8 * e + 3]),
                                                    pack_bf16x2(x[8 * e + 4], x[8 * e + 5]),
                                                    pack_bf16x2(x[8 * e + 6], x[8 * e + 7]));
                        }
                    }
                    if (live && t == 0) {
                        const float lse2 = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
                        if (part)
                            ws_lse[prow] = lse2;  // log2 units
                        else if (lse != nullptr)
                            lse[((size_t)b * Hq + h) * S + i] = lse2 * 0.69314718055994531f;
                    }
                }
            } else if (ok && SPLIT && !direct) {
                // segment result: normalised O (fp32) and LSE in log2 units; an empty segment
                // (this tile has no key tile in it) writes O = 0 and LSE = -inf
                if (active) tc_fence_after();
                const bool live = i < S;
                const float inv = (active && l > 0.f) ? osc / l : 0.f;
                const size_t prow = (size_t)blockIdx.x * RB + t * BM + r;
#pragma unroll 1
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t ov[32];
                    if (active) tmem_ld32(tO + c * 32, ov);
                    if (!live) continue;
                    float4 *dst = reinterpret_cast<float4 *>(ws_o + prow * HD + c * 32);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = active ? make_float4(__uint_as_float(ov[4 * e]) * inv,
                                                      __uint_as_float(ov[4 * e + 1]) * inv,
                                                      __uint_as_float(ov[4 * e + 2]) * inv,
                                                      __uint_as_float(ov[4 * e + 3]) * inv)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (live) ws_lse[prow] = (active && l > 0.f) ? m_ref + log2f(l) : -INFINITY;
            } else if (ok) {
                // an inactive tile (its rows see no key) writes O = 0 and LSE = -inf
                if (active) tc_fence_after();
                const bool live = i < S;
                const float inv = (active && l > 0.f) ? osc / l : 0.f;
                const size_t orow = ((size_t)b * Hq + h) * S + (live ? i : 0);
                const long long obase = b * o_sb + h * o_sh + (long long)(live ? i : 0) * o_ss;
#pragma unroll 1
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t ov[32];
                    if (active)
                        tmem_ld32(tO + c * 32, ov);
                    else
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = 0u;
                    if (!live) continue;
                    if (OUT_F32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) +
                                                                 obase + c * 32);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[e] = make_float4(__uint_as_float(ov[4 * e]) * inv,
                                                 __uint_as_float(ov[4 * e + 1]) * inv,
                                                 __uint_as_float(ov[4 * e + 2]) * inv,
                                                 __uint_as_float(ov[4 * e + 3]) * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out) +
                                                               obase + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint32_t w[4];
#pragma unroll
                            for (int f = 0; f < 4; ++f)
                                w[f] = pack_bf16x2(__uint_as_float(ov[8 * e + 2 * f]) * inv,
                                                   __uint_as_float(ov[8 * e + 2 * f + 1]) * inv);
                            dst[e] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (live && lse != nullptr)
                    lse[orow] = (active && l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994531f
                                                    : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *abort_flag) atomicOr(status, 2u);
    if (SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Combine the key segments of each query row (split mode): one warp per row, HD / 32 dims per
// lane; segment weights 2^(lse_s - M), M = max_s lse_s, in segment order. O is written with the
// strides of the kernel above, the LSE as [B, Hq, S].
template <int HD, bool OUT_F32>
__global__ void __launch_bounds__(256)
    prefill_split_merge_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_lse,
                               void *__restrict__ out, float *__restrict__ lse, int B, int S,
                               int Hq, int causal, int J, long long o_sb, long long o_ss,
                               long long o_sh, int NS, int RB)
{
    constexpr int DPL = HD / 32;  // dims per lane: 4 or 2
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const long long row = (long long)blockIdx.x * 8 + warp;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (row >= (long long)B * Hq * S) return;
    const int i = (int)(row % S);
    const int hb = (int)(row / S);  // b * Hq + h
    const int n_rb = (S + RB - 1) / RB;
    const int rb = i / RB, rloc = i % RB;
    const int first = (n_rb - 1 - rb) * NS * Hq * B;  // first block of row block rb
    const int nseg = rb_segments(rb, S, causal, J, RB);
    if (nseg == 1) return;  // that row block wrote its result itself
    // every load of the row in one round: segment LSEs and this lane's dims of each O
    float ls[8];
    float4 x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        ls[k] = -INFINITY;
        x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < nseg) {
            const size_t item = (size_t)first + (size_t)k * Hq * B + hb;
            ls[k] = ws_lse[item * RB + rloc];
            const float *src = ws_o + (item * RB + rloc) * HD + lane * DPL;
            if constexpr (DPL == 4) {
                x[k] = *reinterpret_cast<const float4 *>(src);
            } else {
                const float2 y = *reinterpret_cast<const float2 *>(src);
                x[k] = make_float4(y.x, y.y, 0.f, 0.f);
            }
        }
    }
    float M = ls[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) M = fmaxf(M, ls[k]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float w = ex2(ls[k] - Mu);  // 0 for absent segments
        L += w;
        acc.x = fmaf(w, x[k].x, acc.x);
        acc.y = fmaf(w, x[k].y, acc.y);
        acc.z = fmaf(w, x[k].z, acc.z);
        acc.w = fmaf(w, x[k].w, acc.w);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const size_t orow = (size_t)row;
    const int b = hb / Hq, h = hb % Hq;
    const long long obase = b * o_sb + h * o_sh + (long long)i * o_ss + lane * DPL;
    if (OUT_F32) {
        float *dst = static_cast<float *>(out) + obase;
        if constexpr (DPL == 4)
            *reinterpret_cast<float4 *>(dst) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        else
            *reinterpret_cast<float2 *>(dst) = make_float2(acc.x * inv, acc.y * inv);
    } else {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(out) + obase;
        if constexpr (DPL == 4) {
            uint2 w2;
            w2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            w2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2 *>(dst) = w2;
        } else {
            *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc.x * inv, acc.y * inv);
        }
    }
    if (lse != nullptr && lane == 0)
        lse[orow] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

// V (bf16, element (b, g, r, d) at v + b sb + r ss + g sh + d) -> a contiguous fp16 copy
// [B, Hkv, rows, HD] for the P V product (WRITE = true; WRITE = false only measures, for the
// on-chip conversion). The copy is made with scale 1, which is exact for the usual range of V;
// each block also records the largest finite |v| it saw in each (b, g) slab,
// vmax[(b * Hkv + g) * gridDim.x + blockIdx.x] (bf16 magnitude bits), from which
// v_scale_kernel picks the slab's scale and redoes the slabs that need another one.
// With kv_lens, rows at or past a sequence's key count are written as 0 up to the end of their
// 128-row key tile (the attention kernel reads whole tiles, and 0 * NaN from a stale cache row
// would not be 0) and do not count towards the maximum; later tiles are never read and are
// skipped. Grid: x blocks stride over one (b, g) slab, y over the slabs.
template <int HD, bool WRITE>
__global__ void __launch_bounds__(256)
    convert_v_kernel(const __nv_bfloat16 *__restrict__ v, long long sb, long long ss,
                     long long sh, uint4 *__restrict__ v16, int B, int Hkv, int rows,
                     const int *__restrict__ kv_lens, int max_kv, unsigned *__restrict__ vmax)
{
    constexpr int CPR = HD / 8;  // 16-byte chunks per row
    constexpr int LOG = HD == 128 ? 4 : 3;
    __shared__ uint32_t red[8];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int nbg = B * Hkv;
    for (int bg = blockIdx.y; bg < nbg; bg += gridDim.y) {
        const int b = bg / Hkv, g = bg - b * Hkv;
        int L = rows;
        if (kv_lens != nullptr) {
            L = kv_lens[b];
            L = L < 0 ? 0 : (L > max_kv ? max_kv : L);
        }
        const long long lim = (long long)min((L + 127) & ~127, rows) * CPR;
        const __nv_bfloat16 *src = v + b * sb + g * sh;
        uint4 *dst = v16 + (long long)bg * rows * CPR;
        uint32_t acc = 0;
        for (long long i = blockIdx.x * 256LL + threadIdx.x; i < lim;
             i += (long long)gridDim.x * 256) {
            const long long r = i >> LOG;
            const int c = (int)(i & (CPR - 1));
            uint4 w = make_uint4(0, 0, 0, 0);
            if (r < L) {
                w = *reinterpret_cast<const uint4 *>(src + r * ss + c * 8);
                acc = absmax_acc(acc, w);
                w.x = bf16x2_to_f16x2(w.x);
                w.y = bf16x2_to_f16x2(w.y);
                w.z = bf16x2_to_f16x2(w.z);
                w.w = bf16x2_to_f16x2(w.w);
            }
            if (WRITE) dst[i] = w;
        }
        uint32_t m = max(acc & 0xFFFFu, acc >> 16);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
#pragma unroll
            for (int w2 = 1; w2 < 8; ++w2) m = max(m, red[w2]);
            vmax[(size_t)bg * gridDim.x + blockIdx.x] = m;
        }
        __syncthreads();
    }
}

// Picks the scale 2^-e of V slab bg = blockIdx.x (+ multiples of gridDim.x) from the xconv block
// maxima convert_v_kernel recorded, writes e to vexp[bg], and with `redo` converts a slab whose
// e is not 0 again, as v * 2^-e, into the fp16 copy (that takes the whole block a while, but only
// a V beyond the fp16 range needs it). One block per slab keeps the grid small: its blocks hold
// their SMs while they wait for the conversion kernel (this grid is its programmatic
// dependent), and the attention kernel, launched the same way after this one, needs those SMs.
template <int HD>
__global__ void __launch_bounds__(256)
    v_scale_kernel(const __nv_bfloat16 *__restrict__ v, long long sb, long long ss, long long sh,
                   uint4 *__restrict__ v16, int B, int Hkv, int rows,
                   const int *__restrict__ kv_lens, int max_kv,
                   const unsigned *__restrict__ vmax, int xconv, int *__restrict__ vexp,
                   int redo)
{
    constexpr int CPR = HD / 8;
    constexpr int LOG = HD == 128 ? 4 : 3;
    __shared__ uint32_t red[8];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nbg = B * Hkv;
    for (int bg = blockIdx.x; bg < nbg; bg += gridDim.x) {
        uint32_t m = 0;
        for (int t = threadIdx.x; t < xconv; t += 256) m = max(m, vmax[(size_t)bg * xconv + t]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
#pragma unroll
        for (int w2 = 0; w2 < 8; ++w2) m = max(m, red[w2]);
        __syncthreads();
        const int e = v_scale_exponent(m);
        if (threadIdx.x == 0) vexp[bg] = e;
        if (!redo || e == 0) continue;
        const int b = bg / Hkv, g = bg - b * Hkv;
        int L = rows;
        if (kv_lens != nullptr) {
            L = kv_lens[b];
            L = L < 0 ? 0 : (L > max_kv ? max_kv : L);
        }
        const float s = exp2i(-e);
        const long long lim = (long long)min((L + 127) & ~127, rows) * CPR;
        const __nv_bfloat16 *src = v + b * sb + g * sh;
        uint4 *dst = v16 + (long long)bg * rows * CPR;
        for (long long i = threadIdx.x; i < lim; i += 256) {
            const long long r = i >> LOG;
            const int c = (int)(i & (CPR - 1));
            uint4 w = make_uint4(0, 0, 0, 0);
            if (r < L) {
                w = *reinterpret_cast<const uint4 *>(src + r * ss + c * 8);
                w.x = bf16x2_to_f16x2_scaled(w.x, s);
                w.y = bf16x2_to_f16x2_scaled(w.y, s);
                w.z = bf16x2_to_f16x2_scaled(w.z, s);
                w.w = bf16x2_to_f16x2_scaled(w.w, s);
            }
            dst[i] = w;
        }
    }
}

}  // namespace

// Grid of the V conversion kernel for nbg slabs of `rows` rows of head dim D on `sms` SMs:
// about 8 blocks of 256 threads per SM in all. v_scale_kernel reads its gx block maxima.
void prefill_conv_grid(int nbg, int rows, int D, int sms, int *gx, int *gy)
{
    const int y = nbg < 65535 ? nbg : 65535;
    const long long per = ((long long)rows * (D / 8) + 255) / 256;  // blocks per slab
    long long x = (8LL * (sms > 0 ? sms : 1) + y - 1) / y;
    if (x > per) x = per;
    if (x < 1) x = 1;
    *gx = (int)x;
    *gy = y;
}

namespace {

// The kernels before the attention kernel: the fp16 copy of V with scale 1 (without a copy, only
// the maxima), then the per-slab scale (v_scale_kernel, a programmatic dependent of the first).
// The attention kernel is launched as a programmatic dependent of v_scale_kernel.
cudaError_t launch_v_prep(const PrefillTcArgs &a, cudaStream_t st)
{
    int gx = 1, gy = 1;
    prefill_conv_grid(a.B * a.Hkv, a.v_rows, a.D, a.sms, &gx, &gy);
    const dim3 grid((unsigned)gx, (unsigned)gy);
    const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(a.v_src);
    uint4 *dst = static_cast<uint4 *>(a.v16);
    if (a.D == 128) {
        if (a.vpre)
            convert_v_kernel<128, true><<<grid, 256, 0, st>>>(src, a.v_sb, a.v_ss, a.v_sh, dst,
                                                              a.B, a.Hkv, a.v_rows, a.kv_lens,
                                                              a.max_kv, a.vmax);
        else
            convert_v_kernel<128, false><<<grid, 256, 0, st>>>(src, a.v_sb, a.v_ss, a.v_sh, dst,
                                                               a.B, a.Hkv, a.v_rows, a.kv_lens,
                                                               a.max_kv, a.vmax);
    } else {
        if (a.vpre)
            convert_v_kernel<64, true><<<grid, 256, 0, st>>>(src, a.v_sb, a.v_ss, a.v_sh, dst,
                                                             a.B, a.Hkv, a.v_rows, a.kv_lens,
                                                             a.max_kv, a.vmax);
        else
            convert_v_kernel<64, false><<<grid, 256, 0, st>>>(src, a.v_sb, a.v_ss, a.v_sh, dst,
                                                              a.B, a.Hkv, a.v_rows, a.kv_lens,
                                                              a.max_kv, a.vmax);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    const int nbg = a.B * a.Hkv;
    cfg.gridDim = dim3((unsigned)(nbg < 65535 ? nbg : 65535));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, a.D == 128 ? v_scale_kernel<128> : v_scale_kernel<64>, src,
                              a.v_sb, a.v_ss, a.v_sh, dst, a.B, a.Hkv, a.v_rows, a.kv_lens,
                              a.max_kv, (const unsigned *)a.vmax, gx, a.vexp, a.vpre);
}

template <int HD, bool OUT_F32, bool SPLIT, bool VPRE, bool PAIR>
cudaError_t launch_t(const PrefillTcArgs &a, cudaStream_t st)
{
    constexpr auto kern = prefill_tc_kernel<HD, OUT_F32, SPLIT, VPRE, PAIR>;
    static bool attr_set[64] = {};  // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Geo<HD>::kSmem);
        if (e != cudaSuccess) return e;
        // the warpgroups' register split assumes exactly kRegsLaunch registers per thread
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
        if (dev < 64) attr_set[dev] = true;
    }
    constexpr int RB = PAIR ? BM : 2 * BM;
    const int n_rb = (a.S + RB - 1) / RB;
    long long blocks = (long long)n_rb * a.Hq * a.B;
    const int NS = SPLIT ? split_slots(a.S, a.causal, a.J, RB) : 1;
    if (SPLIT) blocks = (long long)n_rb * NS * a.Hq * a.B;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    e = launch_v_prep(a, st);
    if (e != cudaSuccess) return e;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = Geo<HD>::kSmem;
        cfg.stream = st;
        cfg.attrs = pdl;
        cfg.numAttrs = 1;  // starts while the V kernels finish
        e = cudaLaunchKernelEx(&cfg, kern, a.tq, a.tk, a.tv, a.o, a.lse, a.B, a.S, a.Hq, a.Hkv,
                               a.scale_log2, a.causal, a.status, a.J, a.ws_o, a.ws_lse, a.kv_lens,
                               a.kv_lens ? a.max_kv : a.S, a.front, a.o_sb, a.o_ss, a.o_sh, NS,
                               (const int *)a.vexp, wait_limit_cycles());
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess || !SPLIT) return e;
    const long long rows = (long long)a.B * a.Hq * a.S;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_split_merge_kernel<HD, OUT_F32>, (const float *)a.ws_o,
                              (const float *)a.ws_lse, a.o, a.lse, a.B, a.S, a.Hq, a.causal, a.J,
                              a.o_sb, a.o_ss, a.o_sh, NS, RB);
}

template <int HD, bool PAIR>
cudaError_t launch_hp(const PrefillTcArgs &a, bool out_f32, cudaStream_t st)
{
    // the key split always has scratch, so it always has the fp16 copy of V as well
    if (a.J > 0)
        return out_f32 ? launch_t<HD, true, true, true, PAIR>(a, st)
                       : launch_t<HD, false, true, true, PAIR>(a, st);
    if (a.vpre)
        return out_f32 ? launch_t<HD, true, false, true, PAIR>(a, st)
                       : launch_t<HD, false, false, true, PAIR>(a, st);
    return out_f32 ? launch_t<HD, true, false, false, PAIR>(a, st)
                   : launch_t<HD, false, false, false, PAIR>(a, st);
}

template <int HD>
cudaError_t launch_hd(const PrefillTcArgs &a, bool out_f32, cudaStream_t st)
{
    return a.pair ? launch_hp<HD, true>(a, out_f32, st) : launch_hp<HD, false>(a, out_f32, st);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillTcArgs &a, bool out_f32, cudaStream_t st)
{
    if (a.D == 64) return launch_hd<64>(a, out_f32, st);
    if (a.D == 128) return launch_hd<128>(a, out_f32, st);
    return cudaErrorInvalidValue;
}

size_t prefill_split_plan(int B, int S, int Hq, int D, int causal, int num_sms, int *pair_out,
                          int *J_out)
{
    constexpr int RB = 2 * BM;  // rows per block of the plain (two-tile) blocks
    // Splitting the key range of the long (causal: the late) row blocks into segments of J key
    // tiles evens out the blocks' work when the grid is only a few waves deep. The choice is an
    // estimate of the finishing time: blocks (one per SM at a time, heaviest first, as launched)
    // are list-scheduled on the SMs at a cost of their key tiles plus a fixed start-up and
    // write-out cost, plus the traffic of the partial results of the split row blocks and the
    // merge launch. Row blocks left in one segment write their result directly. At most 8
    // segments per row block (the merge kernel reads up to 8).
    *J_out = 0;
    *pair_out = 0;
    const int n_rb = (S + RB - 1) / RB;
    const long long heads = (long long)Hq * B;
    // A grid of two-tile blocks that fits in one wave of SMs: pair mode instead, 128 rows per
    // block, whose two softmax warpgroups take the key tiles in turns (the heaviest row block's
    // chain of key steps is cut in two inside the block, with no partials and no merge kernel).
    // Measured at one wave or less it beats every key split (B1 S2048 25.6 vs 31.7 us, B1 S4096
    // 42.0 vs 50.2, B2 S2048 31.7 vs 35.8); at two waves it loses (B1 S8192 126 vs 101), and
    // pair blocks with a key split never won.
    if (num_sms > 0 && (long long)n_rb * heads <= num_sms) {
        *pair_out = 1;
        return 0;
    }
    if ((long long)n_rb * heads >= 4LL * num_sms || num_sms <= 0) return 0;
    static std::mutex mu;
    static std::map<std::array<long long, 6>, int> cache;
    const std::array<long long, 6> key = {B, S, Hq, D, causal, num_sms};
    int best = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            best = it->second;
        } else {
            // Cost model in key-tile steps (one step about 1.9 us), fitted to measured
            // B1-B2 S2048-8192 causal timings over several split lengths: a block costs its
            // steps plus 4 (start-up: TMEM, barriers, Q and first K/V loads; write-out); a
            // split adds about 2 steps (merge launch and dependency wait) and 1e-4 step per
            // row of a split row block (partials written, read back and merged).
            constexpr double kStart = 4.0;
            constexpr double kMerge = 2.1;
            constexpr double kRowSteps = 1.05e-4;
            int nmax = 0;
            for (int rb = 0; rb < n_rb; ++rb) nmax = std::max(nmax, rb_key_tiles(rb, S, causal, RB));
            std::vector<double> load;
            auto estimate = [&](int J) {
                load.assign(num_sms, 0.0);
                std::priority_queue<double, std::vector<double>, std::greater<double>> q(
                    load.begin(), load.end());
                double rows_split = 0.0;
                for (int rb = n_rb - 1; rb >= 0; --rb) {
                    const int t = rb_key_tiles(rb, S, causal, RB);
                    const int ns = J > 0 ? (t + J - 1) / J : 1;
                    if (ns > 1) rows_split += 2.0 * BM * heads * ns;
                    for (int k = 0; k < ns; ++k) {
                        const int len = J > 0 ? std::min(J, t - k * J) : t;
                        for (long long h = 0; h < heads; ++h) {
                            const double at = q.top();
                            q.pop();
                            q.push(at + len + kStart);
                        }
                    }
                }
                double end = 0.0;
                while (!q.empty()) {
                    end = std::max(end, q.top());
                    q.pop();
                }
                return end + (J > 0 ? kMerge : 0.0) + rows_split * kRowSteps;
            };
            // a split must promise a tenth off the unsplit estimate (the model's error is a
            // few percent)
            const double plain = estimate(0);
            double best_t = 0.9 * plain;
            for (int J = std::max(2, (nmax + 7) / 8); J < nmax; ++J) {
                const double t = estimate(J);
                if (t < best_t) {
                    best_t = t;
                    best = J;
                }
            }
            cache[key] = best;
        }
    }
    if (best == 0) return 0;
    *J_out = best;
    const long long blocks = (long long)n_rb * split_slots(S, causal, best, RB) * heads;
    return (size_t)blocks * RB * (D + 1) * sizeof(float);
}

}  // namespace gqa
