// decode_noalloc.cu -- single-token decode whose scratch lives in a fixed device array, for
// callers that must not allocate device memory at all.
//
// Who needs this: code that runs where cudaMalloc is not an option -- inside a custom memory
// manager that owns every byte of the device, in a process whose allocator is frozen after
// start-up, or in a plug-in that is handed buffers but no allocator. The regular decode entry
// points either grow a library-owned buffer with cudaMalloc or take a caller workspace; this
// one needs neither.
//
// The split-KV decode kernels write their per-chunk partial results (running max, sum and
// unnormalised output per query head) to scratch memory, and the merge kernel reads them back.
// Here that scratch is g_noalloc_scratch below: a file-scope device array of
// ATTN_DECODE_NOALLOC_SCRATCH_BYTES bytes that every GPU loading the library holds until the
// process exits. For batches up to 1024 the split kernel runs on as many warps as the array has
// room for; shapes that do not fit even so are rejected.
//
// Host code cannot use the array's name as a device pointer, so the first call on each device
// looks its address up with cudaGetSymbolAddress (with that device current) and keeps it.
#include "gqa_attn.h"
#include "internal.h"

#include <cmath>
#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device (looked up once per device).
int scratch_address(void **out)
{
    static void *addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return ATTN_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" int attn_decode_noalloc(const void *q, const void *kcache, const void *vcache,
                                   const int *seqlens, void *o, float *lse, int B, int Hq,
                                   int Hkv, int D, int max_len, float scale, int out_dtype,
                                   void *stream)
{
    if (!q || !kcache || !vcache || !seqlens || !o) return ATTN_ERR_INVALID;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_len <= 0 || Hq % Hkv != 0)
        return ATTN_ERR_INVALID;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID;
    if (out_dtype != ATTN_F32 && out_dtype != ATTN_BF16) return ATTN_ERR_INVALID;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || Hq > 65535) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o))
        return ATTN_ERR_ALIGN;
    if (!aligned4(seqlens) || (lse && !aligned4(lse))) return ATTN_ERR_ALIGN;

    // The stream kernel's partials grow with its warp count: launch only as many warps as the
    // array has room for (the chunked kernel for large batches needs its full size).
    const int warps = gqa::decode_warps_within(B, Hq, Hkv, D, max_len,
                                               (size_t)ATTN_DECODE_NOALLOC_SCRATCH_BYTES);
    if (warps <= 0) return ATTN_ERR_WORKSPACE;

    void *ws = nullptr;
    int rc = scratch_address(&ws);
    if (rc != ATTN_OK) return rc;
    gqa::DecodeArgs a;
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
    // Nothing needs clearing: every partial result the merge kernel reads was written by the
    // split kernel of the same call.
    a.ws = ws;
    a.max_warps = warps;
    a.scale_log2 = scale * 1.4426950408889634f;
    rc = gqa::status_word_ptr(&a.status);
    if (rc != ATTN_OK) return rc;
    const cudaError_t e = gqa::launch_decode(a, out_dtype == ATTN_F32,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
