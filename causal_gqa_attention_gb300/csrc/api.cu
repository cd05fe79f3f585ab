// api.cu -- the C ABI declared in include/gqa_attn.h: host-side argument checks, tensor-map
// encoding for the TMA loads, the library-owned decode workspace and the device status word.
// Every check runs before the first CUDA call, so a rejected call touches no GPU state.
#include "gqa_attn.h"
#include "internal.h"

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

// Per-device status word written by the kernels (bits ATTN_DEV_*).
__device__ unsigned int g_attn_status;

namespace {
// Bound on each pipeline wait, in SM clock cycles (about 2 s at 2 GHz), passed to every launch;
// attn_debug_set_wait_limit changes it for later launches.
constexpr long long kDefaultWaitLimit = 4000000000LL;
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
}  // namespace

namespace {

using gqa::DecodeArgs;
using gqa::PrefillTcArgs;

constexpr int kMaxDevices = 64;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

// ---- driver entry point for tensor-map encoding (no link-time dependency on libcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Element strides of one [B, H, rows, D] operand: batch, row (token), head; the head dim is
// contiguous.
struct Strides {
    long long b, s, h;
};

Strides contiguous(int H, long long rows, int D)
{
    return Strides{(long long)H * rows * D, D, rows * D};
}

// 16-bit tensor (bf16, or fp16 with f16 = true) viewed as {D, rows, heads, batch} with the
// given element strides, a 64-column x 128-row box and 128-byte swizzle; reads past `rows` (or
// any extent) fill with zeros.
bool encode_bf16_4d(CUtensorMap *m, const void *base, int D, long long rows, int heads, int batch,
                    const Strides &st, bool f16 = false)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads,
                                (cuuint64_t)batch};
    const cuuint64_t strides[3] = {(cuuint64_t)st.s * 2, (cuuint64_t)st.h * 2,
                                   (cuuint64_t)st.b * 2};  // bytes, dims 1..3
    const cuuint32_t box[4] = {64, 128, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Strides usable by the tensor maps (bf16 operands) or by the 16-byte output stores: positive,
// below 2^39 elements, and a multiple of 16 bytes.
bool strides_ok(const Strides &st, int elem_bytes)
{
    const long long v[3] = {st.b, st.s, st.h};
    for (long long x : v)
        if (x <= 0 || x >= (1LL << 39) || (x * elem_bytes) % 16 != 0) return false;
    return true;
}

// ---- device status word address, per device
int status_ptr(unsigned **out)
{
    static unsigned *ptrs[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess) return ATTN_ERR_CUDA;
        ptrs[dev] = static_cast<unsigned *>(p);
    }
    *out = ptrs[dev];
    return ATTN_OK;
}

// ---- library-owned scratch, per device. Growing it allocates a new buffer and keeps the old
// one for the life of the process: a CUDA graph captured with the old buffer keeps replaying on
// valid memory, and no kernel still in flight can see its buffer freed. Sizes at least double,
// so the retained buffers add up to less than the current one.
struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
    std::vector<void *> retired;
};
Workspace g_ws[kMaxDevices];
std::mutex g_ws_mu;

int workspace_acquire(size_t need, cudaStream_t stream, bool may_grow, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace &w = g_ws[dev];
    if (w.bytes < need) {
        if (!may_grow) return ATTN_ERR_WORKSPACE;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return ATTN_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return ATTN_ERR_WORKSPACE;
        size_t sz = need < (1u << 20) ? (1u << 20) : need;
        if (sz < 2 * w.bytes) sz = 2 * w.bytes;
        void *p = nullptr;
        if (cudaMalloc(&p, sz) != cudaSuccess) return ATTN_ERR_CUDA;
        if (w.ptr) w.retired.push_back(w.ptr);
        w.ptr = p;
        w.bytes = sz;
    }
    *out = w.ptr;
    return ATTN_OK;
}

int sm_count(int *out)
{
    static int cached[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        cached[dev] = n;
    }
    *out = cached[dev];
    return ATTN_OK;
}

// Largest fp16 copy of V a prefill call makes in its scratch; larger calls convert V on chip
// instead.
constexpr size_t kMaxV16Bytes = size_t(1) << 30;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Scratch of one tensor-core prefill call, in this order, each part 256-byte aligned: the V
// scale area (per-slab exponents, then the conversion blocks' maxima; always needed), the key
// split's partial results (0 = no split) and the fp16 copy of V (0 = V is converted on chip).
struct PrefillScratch {
    size_t nbg = 0, gx = 0;
    size_t small = 0, split = 0, v16 = 0;
    size_t split_rows = 0;  // rows of partial results (blocks x rows per block)
};

PrefillScratch prefill_scratch_sizes(int B, int Hkv, int rows, int D, int sms, size_t split_bytes)
{
    int gx = 1, gy = 1;
    gqa::prefill_conv_grid(B * Hkv, rows, D, sms, &gx, &gy);
    PrefillScratch p;
    p.nbg = (size_t)B * Hkv;
    p.gx = (size_t)gx;
    p.small = align256(p.nbg * sizeof(int)) + align256(p.nbg * p.gx * sizeof(unsigned));
    p.split = align256(split_bytes);
    p.split_rows = split_bytes / ((size_t)(D + 1) * sizeof(float));
    const size_t v16 = p.nbg * (size_t)rows * D * 2;
    p.v16 = v16 <= kMaxV16Bytes ? v16 : 0;
    return p;
}

// Places one call's scratch, trying in turn: split + fp16 copy, the copy alone, neither (V
// converted on chip; the split needs the copy). It goes in the caller's workspace when one is
// given (the first arrangement that fits), else in the library-owned buffer, grown when that is
// possible (not during stream capture). Sets a.J, a.ws_o / a.ws_lse, a.vpre / a.v16 and
// a.vexp / a.vmax. ATTN_ERR_WORKSPACE when not even the V scale area fits.
int prefill_scratch(PrefillTcArgs &a, int J, const PrefillScratch &p, void *caller,
                    size_t caller_bytes, cudaStream_t st)
{
    struct Option {
        bool split, v16;
    };
    const Option opts[3] = {{true, true}, {false, true}, {false, false}};
    for (const Option &o : opts) {
        if (o.split && (J == 0 || p.split == 0)) continue;
        if (o.v16 && p.v16 == 0) continue;
        const size_t need = p.small + (o.split ? p.split : 0) + (o.v16 ? p.v16 : 0);
        void *ws = nullptr;
        if (caller != nullptr) {
            if (caller_bytes < need) continue;
            ws = caller;
        } else {
            const int rc = workspace_acquire(need, st, true, &ws);
            if (rc == ATTN_ERR_WORKSPACE) continue;
            if (rc != ATTN_OK) return rc;
        }
        uint8_t *base = static_cast<uint8_t *>(ws);
        a.vexp = reinterpret_cast<int *>(base);
        a.vmax = reinterpret_cast<unsigned *>(base + align256(p.nbg * sizeof(int)));
        size_t off = p.small;
        a.J = 0;
        a.vpre = 0;
        if (o.split) {
            a.J = J;
            a.ws_o = reinterpret_cast<float *>(base + off);
            a.ws_lse = a.ws_o + p.split_rows * a.D;
            off += p.split;
        }
        if (o.v16) {
            a.vpre = 1;
            a.v16 = base + off;
        }
        return ATTN_OK;
    }
    return ATTN_ERR_WORKSPACE;
}

int check_prefill(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                  int S, int Hq, int Hkv, int D, float scale, int in_t, int out_t)
{
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID;
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID;
    if (!scale_ok(scale)) return ATTN_ERR_INVALID;
    if ((in_t != ATTN_F32 && in_t != ATTN_BF16) || (out_t != ATTN_F32 && out_t != ATTN_BF16))
        return ATTN_ERR_INVALID;
    if ((long long)B * Hq > (1LL << 30) || (long long)B * Hq * S > (1LL << 40))
        return ATTN_ERR_UNSUPPORTED;
    if (in_t == ATTN_BF16 && D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (in_t == ATTN_BF16 && (long long)((S + 255) / 256) * B * Hq >= (1LL << 31))
        return ATTN_ERR_UNSUPPORTED;
    if (in_t == ATTN_F32 && ((D != 64 && D != 128) || out_t != ATTN_F32)) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_ALIGN;
    if (lse && !aligned4(lse)) return ATTN_ERR_ALIGN;
    if (in_t == ATTN_F32 && (Hq > 65535 || B > 65535)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

int check_decode(const void *q, const void *kc, const void *vc, const int *seqlens, void *o,
                 float *lse, int B, int Hq, int Hkv, int D, int max_len, float scale, int out_t)
{
    if (!q || !kc || !vc || !seqlens || !o) return ATTN_ERR_INVALID;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_len <= 0 || Hq % Hkv != 0)
        return ATTN_ERR_INVALID;
    if (!scale_ok(scale)) return ATTN_ERR_INVALID;
    if (out_t != ATTN_F32 && out_t != ATTN_BF16) return ATTN_ERR_INVALID;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || (long long)Hkv * (Hq / Hkv) > 65535) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(o)) return ATTN_ERR_ALIGN;
    if (!aligned4(seqlens) || (lse && !aligned4(lse))) return ATTN_ERR_ALIGN;
    return ATTN_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// bf16 prefill on the tensor-core kernel for checked arguments and strides; scratch in `ws`
// (ws_bytes) or, with ws == nullptr, in the library-owned buffer.
int prefill_bf16(const void *q, const void *k, const void *v, void *o, float *lse, int B, int S,
                 int Hq, int Hkv, int D, float scale, int causal, int out_dtype, const Strides &qs,
                 const Strides &ks, const Strides &vs, const Strides &os, void *ws,
                 size_t ws_bytes, void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PrefillTcArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!encode_bf16_4d(&a.tq, q, D, S, Hq, B, qs) || !encode_bf16_4d(&a.tk, k, D, S, Hkv, B, ks) ||
        !encode_bf16_4d(&a.tv, v, D, S, Hkv, B, vs))
        return ATTN_ERR_CUDA;
    a.o = o;
    a.o_sb = os.b;
    a.o_ss = os.s;
    a.o_sh = os.h;
    a.lse = lse;
    a.B = B;
    a.S = S;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.causal = causal ? 1 : 0;
    int rc = status_ptr(&a.status);
    if (rc != ATTN_OK) return rc;
    // Small grids (fewer row blocks x heads than SMs) split the keys of each row block over
    // several blocks and merge; the partials use the scratch, as does the fp16 copy of V.
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != ATTN_OK) return rc;
    a.sms = sms;
    int J = 0, pair = 0;
    const size_t need = gqa::prefill_split_plan(B, S, Hq, D, causal ? 1 : 0, sms, &pair, &J);
    a.pair = pair;
    rc = prefill_scratch(a, J, prefill_scratch_sizes(B, Hkv, S, D, sms, need), ws, ws_bytes, st);
    if (rc != ATTN_OK) return rc;
    a.v_src = v;
    a.v_sb = vs.b;
    a.v_ss = vs.s;
    a.v_sh = vs.h;
    a.v_rows = S;
    if (a.vpre &&
        !encode_bf16_4d(&a.tv, a.v16, D, S, Hkv, B, contiguous(Hkv, S, D), true))
        return ATTN_ERR_CUDA;
    return cuda_status(gqa::launch_prefill_tc(a, out_dtype == ATTN_F32, st));
}

}  // namespace

namespace gqa {
int status_word_ptr(unsigned **out) { return status_ptr(out); }
long long wait_limit_cycles() { return g_wait_limit.load(); }
}  // namespace gqa

extern "C" {

int attn_version(void) { return 100; }

int attn_debug_build(void)
{
#ifdef GQA_ATTN_DEBUG
    return 1;
#else
    return 0;
#endif
}

const char *attn_status_string(int s)
{
    switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "workspace too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

int attn_prefill_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int S, int Hq, int Hkv, int D, float scale, int causal, int in_dtype,
                    int out_dtype, void *stream)
{
    int rc = check_prefill(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, in_dtype, out_dtype);
    if (rc != ATTN_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (in_dtype == ATTN_F32)
        return cuda_status(gqa::launch_prefill_f32(
            static_cast<const float *>(q), static_cast<const float *>(k),
            static_cast<const float *>(v), static_cast<float *>(o), lse, B, S, Hq, Hkv, D, scale,
            causal ? 1 : 0, st));
    return prefill_bf16(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, out_dtype,
                        contiguous(Hq, S, D), contiguous(Hkv, S, D), contiguous(Hkv, S, D),
                        contiguous(Hq, S, D), nullptr, 0, stream);
}

size_t attn_prefill_workspace_bytes(int B, int S, int Hq, int Hkv, int D, int causal)
{
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || (D != 64 && D != 128))
        return 0;
    int sms = 0;
    if (sm_count(&sms) != ATTN_OK) return 0;
    int J = 0, pair = 0;
    const size_t split = gqa::prefill_split_plan(B, S, Hq, D, causal ? 1 : 0, sms, &pair, &J);
    const PrefillScratch p = prefill_scratch_sizes(B, Hkv, S, D, sms, split);
    return p.small + (J > 0 && p.v16 > 0 ? p.split : 0) + p.v16;
}

int attn_prefill_ws(const void *q, const void *k, const void *v, void *o, float *lse, int B, int S,
                    int Hq, int Hkv, int D, float scale, int causal, int out_dtype,
                    void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_prefill(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, ATTN_BF16, out_dtype);
    if (rc != ATTN_OK) return rc;
    if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return ATTN_ERR_ALIGN;
    return prefill_bf16(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, out_dtype,
                        contiguous(Hq, S, D), contiguous(Hkv, S, D), contiguous(Hkv, S, D),
                        contiguous(Hq, S, D), workspace, workspace_bytes, stream);
}

int attn_prefill_strided(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int S, int Hq, int Hkv, int D, const long long *q_strides,
                         const long long *k_strides, const long long *v_strides,
                         const long long *o_strides, float scale, int causal, int out_dtype,
                         void *stream)
{
    if (!q_strides || !k_strides || !v_strides || !o_strides) return ATTN_ERR_INVALID;
    int rc = check_prefill(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, ATTN_BF16, out_dtype);
    if (rc != ATTN_OK) return rc;
    const Strides qs{q_strides[0], q_strides[1], q_strides[2]};
    const Strides ks{k_strides[0], k_strides[1], k_strides[2]};
    const Strides vs{v_strides[0], v_strides[1], v_strides[2]};
    const Strides os{o_strides[0], o_strides[1], o_strides[2]};
    if (!strides_ok(qs, 2) || !strides_ok(ks, 2) || !strides_ok(vs, 2) ||
        !strides_ok(os, out_dtype == ATTN_F32 ? 4 : 2))
        return ATTN_ERR_ALIGN;
    return prefill_bf16(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, out_dtype, qs, ks, vs,
                        os, nullptr, 0, stream);
}

namespace {
int chunk_or_varlen(const void *q, const void *kc, const void *vc, const int *seqlens, void *o,
                    float *lse, int B, int Sq, int Hq, int Hkv, int D, int max_len, float scale,
                    int causal, int out_dtype, int front, const Strides &qs, const Strides &ks,
                    const Strides &vs, const Strides &os, void *stream);

// Strides from three host int64 arrays {batch, token, head}: ATTN_ERR_INVALID for a NULL array,
// ATTN_ERR_ALIGN for strides the tensor maps or the output stores cannot use.
int read_strides(const long long *qa, const long long *ka, const long long *va,
                 const long long *oa, int out_dtype, Strides *qs, Strides *ks, Strides *vs,
                 Strides *os)
{
    if (!qa || !ka || !va || !oa) return ATTN_ERR_INVALID;
    *qs = Strides{qa[0], qa[1], qa[2]};
    *ks = Strides{ka[0], ka[1], ka[2]};
    *vs = Strides{va[0], va[1], va[2]};
    *os = Strides{oa[0], oa[1], oa[2]};
    if (!strides_ok(*qs, 2) || !strides_ok(*ks, 2) || !strides_ok(*vs, 2) ||
        !strides_ok(*os, out_dtype == ATTN_F32 ? 4 : 2))
        return ATTN_ERR_ALIGN;
    return ATTN_OK;
}
}  // namespace

int attn_prefill_varlen(const void *q, const void *k, const void *v, const int *seqlens, void *o,
                        float *lse, int B, int S, int Hq, int Hkv, int D, float scale, int causal,
                        int out_dtype, void *stream)
{
    return chunk_or_varlen(q, k, v, seqlens, o, lse, B, S, Hq, Hkv, D, S, scale, causal,
                           out_dtype, 1, contiguous(Hq, S, D), contiguous(Hkv, S, D),
                           contiguous(Hkv, S, D), contiguous(Hq, S, D), stream);
}

int attn_prefill_varlen_strided(const void *q, const void *k, const void *v, const int *seqlens,
                                void *o, float *lse, int B, int S, int Hq, int Hkv, int D,
                                const long long *q_strides, const long long *k_strides,
                                const long long *v_strides, const long long *o_strides,
                                float scale, int causal, int out_dtype, void *stream)
{
    Strides qs, ks, vs, os;
    int rc = read_strides(q_strides, k_strides, v_strides, o_strides, out_dtype, &qs, &ks, &vs,
                          &os);
    if (rc != ATTN_OK) return rc;
    return chunk_or_varlen(q, k, v, seqlens, o, lse, B, S, Hq, Hkv, D, S, scale, causal,
                           out_dtype, 1, qs, ks, vs, os, stream);
}

int attn_chunk(const void *q, const void *kcache, const void *vcache, const int *seqlens,
               void *o, float *lse, int B, int Sq, int Hq, int Hkv, int D, int max_len,
               float scale, int causal, int out_dtype, void *stream)
{
    return chunk_or_varlen(q, kcache, vcache, seqlens, o, lse, B, Sq, Hq, Hkv, D, max_len, scale,
                           causal, out_dtype, 0, contiguous(Hq, Sq, D),
                           contiguous(Hkv, max_len, D), contiguous(Hkv, max_len, D),
                           contiguous(Hq, Sq, D), stream);
}

int attn_chunk_strided(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                       void *o, float *lse, int B, int Sq, int Hq, int Hkv, int D, int max_len,
                       const long long *q_strides, const long long *k_strides,
                       const long long *v_strides, const long long *o_strides, float scale,
                       int causal, int out_dtype, void *stream)
{
    Strides qs, ks, vs, os;
    int rc = read_strides(q_strides, k_strides, v_strides, o_strides, out_dtype, &qs, &ks, &vs,
                          &os);
    if (rc != ATTN_OK) return rc;
    return chunk_or_varlen(q, kcache, vcache, seqlens, o, lse, B, Sq, Hq, Hkv, D, max_len, scale,
                           causal, out_dtype, 0, qs, ks, vs, os, stream);
}

}  // extern "C"

namespace {
int chunk_or_varlen(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                    void *o, float *lse, int B, int Sq, int Hq, int Hkv, int D, int max_len,
                    float scale, int causal, int out_dtype, int front, const Strides &qs,
                    const Strides &ks, const Strides &vs, const Strides &os, void *stream)
{
    if (!seqlens) return ATTN_ERR_INVALID;
    if (max_len <= 0) return ATTN_ERR_INVALID;
    int rc = check_prefill(q, kcache, vcache, o, lse, B, Sq, Hq, Hkv, D, scale, ATTN_BF16,
                           out_dtype);
    if (rc != ATTN_OK) return rc;
    if (!aligned4(seqlens)) return ATTN_ERR_ALIGN;
    if ((long long)B * Hkv * max_len > (1LL << 40)) return ATTN_ERR_UNSUPPORTED;
    PrefillTcArgs a;
    std::memset(&a, 0, sizeof(a));
    if (!encode_bf16_4d(&a.tq, q, D, Sq, Hq, B, qs) ||
        !encode_bf16_4d(&a.tk, kcache, D, max_len, Hkv, B, ks) ||
        !encode_bf16_4d(&a.tv, vcache, D, max_len, Hkv, B, vs))
        return ATTN_ERR_CUDA;
    a.o = o;
    a.o_sb = os.b;
    a.o_ss = os.s;
    a.o_sh = os.h;
    a.lse = lse;
    a.B = B;
    a.S = Sq;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.causal = causal ? 1 : 0;
    a.kv_lens = seqlens;
    a.max_kv = max_len;
    a.front = front;
    rc = status_ptr(&a.status);
    if (rc != ATTN_OK) return rc;
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != ATTN_OK) return rc;
    a.sms = sms;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = prefill_scratch(a, 0, prefill_scratch_sizes(B, Hkv, max_len, D, sms, 0), nullptr, 0, st);
    if (rc != ATTN_OK) return rc;
    a.v_src = vcache;
    a.v_sb = vs.b;
    a.v_ss = vs.s;
    a.v_sh = vs.h;
    a.v_rows = max_len;
    if (a.vpre &&
        !encode_bf16_4d(&a.tv, a.v16, D, max_len, Hkv, B, contiguous(Hkv, max_len, D), true))
        return ATTN_ERR_CUDA;
    return cuda_status(gqa::launch_prefill_tc(a, out_dtype == ATTN_F32,
                                              static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

int attn_prefill(const void *q, const void *k, const void *v, void *o, float *lse, int B, int S,
                 int Hq, int Hkv, int D, float scale, int causal, void *stream)
{
    return attn_prefill_ex(q, k, v, o, lse, B, S, Hq, Hkv, D, scale, causal, ATTN_BF16, ATTN_BF16,
                           stream);
}

int attn_decode_chunk_len(int B, int Hkv, int max_len)
{
    if (B <= 0 || Hkv <= 0 || max_len <= 0) return 0;
    return gqa::decode_chunk_len(B, Hkv, max_len);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_len <= 0 || Hq % Hkv != 0) return 0;
    return gqa::decode_workspace_bytes(B, Hq, Hkv, D, max_len);
}

int attn_reserve_workspace(int B, int Hq, int Hkv, int D, int max_len)
{
    const size_t need = attn_decode_workspace_bytes(B, Hq, Hkv, D, max_len);
    if (need == 0) return ATTN_ERR_INVALID;
    void *p = nullptr;
    return workspace_acquire(need, nullptr, true, &p);
}

int attn_reserve_workspace_bytes(size_t bytes)
{
    void *p = nullptr;
    return workspace_acquire(bytes, nullptr, true, &p);
}

int attn_decode_ex(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                   void *o, float *lse, int B, int Hq, int Hkv, int D, int max_len, float scale,
                   void *workspace, size_t workspace_bytes, int out_dtype, void *stream)
{
    int rc = check_decode(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, D, max_len, scale,
                          out_dtype);
    if (rc != ATTN_OK) return rc;
    const size_t need = gqa::decode_workspace_bytes(B, Hq, Hkv, D, max_len);
    if (workspace != nullptr) {
        if (workspace_bytes < need) return ATTN_ERR_WORKSPACE;
        if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *ws = workspace;
    if (ws == nullptr) {
        rc = workspace_acquire(need, st, true, &ws);
        if (rc != ATTN_OK) return rc;
    }
    DecodeArgs a;
    a.q = q;
    a.kc = kcache;
    a.vc = vcache;
    a.seqlens = seqlens;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.max_len = max_len;
    a.ws = ws;
    a.scale_log2 = scale * 1.4426950408889634f;
    rc = status_ptr(&a.status);
    if (rc != ATTN_OK) return rc;
    return cuda_status(gqa::launch_decode(a, out_dtype == ATTN_F32, st));
}

int attn_decode_rope(const void *q, const void *k_new, const void *v_new, const float *cos_t,
                     const float *sin_t, void *kcache, void *vcache, const int *seqlens, void *o,
                     float *lse, int B, int Hq, int Hkv, int D, int max_len, float scale,
                     int out_dtype, void *stream)
{
    int rc = check_decode(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, D, max_len, scale,
                          out_dtype);
    if (rc != ATTN_OK) return rc;
    if (!k_new || !v_new || !cos_t || !sin_t) return ATTN_ERR_INVALID;
    if (!aligned16(cos_t) || !aligned16(sin_t) || !aligned16(k_new) || !aligned16(v_new))
        return ATTN_ERR_ALIGN;
    const bool fused = gqa::decode_fuses_rope(B);
    const size_t dec = (gqa::decode_workspace_bytes(B, Hq, Hkv, D, max_len) + 255) & ~(size_t)255;
    const size_t need = dec + (fused ? 0 : (size_t)B * Hq * D * sizeof(float));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    rc = workspace_acquire(need, st, true, &ws);
    if (rc != ATTN_OK) return rc;
    DecodeArgs a;
    if (fused) {
        // one kernel: RoPE of q and of the new key, cache store, attention
        a.q = q;
        a.k_new = k_new;
        a.v_new = v_new;
        a.cos_t = cos_t;
        a.sin_t = sin_t;
    } else {
        float *q_rot = reinterpret_cast<float *>(static_cast<char *>(ws) + dec);
        rc = cuda_status(gqa::launch_rope_append(q, k_new, v_new, cos_t, sin_t, kcache, vcache,
                                                 seqlens, q_rot, B, Hq, Hkv, D, max_len, st));
        if (rc != ATTN_OK) return rc;
        a.q = q_rot;
        a.q_f32 = true;
    }
    a.kc = kcache;
    a.vc = vcache;
    a.seqlens = seqlens;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.max_len = max_len;
    a.ws = ws;
    a.scale_log2 = scale * 1.4426950408889634f;
    rc = status_ptr(&a.status);
    if (rc != ATTN_OK) return rc;
    return cuda_status(gqa::launch_decode(a, out_dtype == ATTN_F32, st));
}

int attn_decode(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                void *o, int B, int Hq, int Hkv, int D, int max_len, float scale, void *stream)
{
    return attn_decode_ex(q, kcache, vcache, seqlens, o, nullptr, B, Hq, Hkv, D, max_len, scale,
                          nullptr, 0, ATTN_BF16, stream);
}

int attn_debug_set_wait_limit(long long cycles)
{
    g_wait_limit.store(cycles > 0 ? cycles : kDefaultWaitLimit);
    return ATTN_OK;
}

int attn_device_status(void *stream, unsigned int *status)
{
    if (!status) return ATTN_ERR_INVALID;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(v)) != cudaSuccess) return ATTN_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
    *status = v;
    return ATTN_OK;
}

}  // extern "C"
