// internal.h -- launchers shared between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gqa {

// Prefill on tcgen05 tensor cores: bf16 q/k/v with head dim 64 or 128. The tensor maps describe
// q as a 4-D bf16 tensor {D, S, Hq, B} and k, v as {D, rows, Hkv, B} (rows = S, or max_kv for a
// cache), each with its own strides, 64 x 128-row boxes and 128-byte swizzle.
struct PrefillTcArgs {
    CUtensorMap tq, tk, tv;  // tv: the fp16 copy of V (vpre != 0) or V itself (bf16)
    void *o;        // bf16 or fp32, element (b, h, i, d) at o + b o_sb + i o_ss + h o_sh + d
    long long o_sb, o_ss, o_sh;
    float *lse;     // [B, Hq, S] or nullptr
    int B, S, Hq, Hkv, D;
    float scale_log2;  // scale * log2(e)
    int causal;
    unsigned *status;  // device status word
    // chunk against a cache: k/v maps view max_kv rows per head; kv_lens[b] keys per sequence
    // (device); the S queries are the last S of them. nullptr: plain prefill (L = S).
    const int *kv_lens = nullptr;
    int max_kv = 0;
    // with kv_lens: 0 = the queries are the last S tokens (cache chunk); 1 = the queries are
    // tokens 0..S-1 of a padded batch, kv_lens[b] of them valid (rows past it are padding)
    int front = 0;
    // small grids: pair != 0 gives each block 128 query rows, its two softmax warpgroups taking
    // the key tiles in turns (combined in the block); J > 0 splits each row block's key tiles
    // into segments of at most J tiles, one block each, partials in ws
    int pair = 0;
    int J = 0;
    float *ws_o = nullptr;    // [blocks, 256, D] fp32
    float *ws_lse = nullptr;  // [blocks, 256] fp32
    // vpre != 0: V is first converted to a contiguous fp16 copy v16 [B, Hkv, v_rows, D] (from
    // v_src, element (b, g, r, d) at v_src + b v_sb + r v_ss + g v_sh + d) and tv maps that
    // copy; vpre == 0: tv maps the bf16 V and the kernel converts it on chip. Required with J.
    int vpre = 0;
    const void *v_src = nullptr;
    long long v_sb = 0, v_ss = 0, v_sh = 0;
    void *v16 = nullptr;
    int v_rows = 0;
    int sms = 0;  // SM count (sizes the conversion grid)
    // V scale per (b, kv head) slab, always required: vmax holds the conversion blocks' maxima
    // ([B * Hkv, gx] of prefill_conv_grid), vexp the chosen exponents [B * Hkv]
    unsigned *vmax = nullptr;
    int *vexp = nullptr;
};
// Grid (gx, gy) of the V conversion kernel for nbg (b, kv head) slabs of `rows` rows.
void prefill_conv_grid(int nbg, int rows, int D, int sms, int *gx, int *gy);
cudaError_t launch_prefill_tc(const PrefillTcArgs &a, bool out_f32, cudaStream_t stream);
// Chooses the small-grid plan for a prefill shape on num_sms SMs: writes pair (0/1) and J
// (0 = no split) and returns the workspace bytes the split needs.
size_t prefill_split_plan(int B, int S, int Hq, int D, int causal, int num_sms, int *pair, int *J);

// Prefill on CUDA cores in fp32 (fp32 q/k/v/o), head dim 64 or 128.
cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, float *o,
                               float *lse, int B, int S, int Hq, int Hkv, int D, float scale,
                               int causal, cudaStream_t stream);

// Decode: a split kernel writes partial (m, l, o) results to the workspace and a merge kernel
// combines them. Batches up to 1024 use the stream kernel (every warp of a persistent grid
// takes an equal slice of all keys), larger ones the chunked kernel (one block per key chunk).
struct DecodeArgs {
    const void *q;        // [B, Hq, D] bf16
    const void *kc, *vc;  // [B, Hkv, max_len, D] bf16
    const int *seqlens;   // [B]
    void *o;              // [B, Hq, D] bf16 or fp32
    float *lse;           // [B, Hq] or nullptr
    void *ws;             // decode_workspace_bytes(...) bytes, 16-byte aligned
    int B, Hq, Hkv, D, max_len;
    float scale_log2;
    unsigned *status;
    bool q_f32 = false;   // q is fp32 (the RoPE step's output) instead of bf16
    // decode with RoPE fused into the stream kernel (batches up to 1024): the new token's key
    // and value [B, Hkv, D] bf16 and the angle tables [max_len, D/2] fp32, all 16-byte aligned;
    // q is then the unrotated bf16 query. nullptr: plain decode.
    const void *k_new = nullptr, *v_new = nullptr;
    const float *cos_t = nullptr, *sin_t = nullptr;
    // at most this many warps for the stream kernel (0: as many as fit on the device); the
    // partials' layout follows the warps actually launched
    int max_warps = 0;
    // filled in by launch_decode for the chunked kernel
    float *ws_o = nullptr;
    float2 *ws_ml = nullptr;
    int chunk = 0, nsplit = 0;
};
cudaError_t launch_decode(const DecodeArgs &a, bool out_f32, cudaStream_t stream);

// Whether launch_decode can fuse RoPE and the cache store into its kernel for batch B (else
// launch_rope_append runs first and the decode reads its fp32 q).
bool decode_fuses_rope(int B);

// RoPE (rotate-half) of the new token of each sequence at position seqlens[b] - 1: q into
// q_rot [B, Hq, D] fp32; k_new rotated and v_new stored at that row of the caches.
cudaError_t launch_rope_append(const void *q, const void *k_new, const void *v_new,
                               const float *cos_t, const float *sin_t, void *kc, void *vc,
                               const int *seqlens, float *q_rot, int B, int Hq, int Hkv, int D,
                               int max_len, cudaStream_t stream);

// Bound on each pipeline wait of the kernels launched from now on, in SM clock cycles: the
// default (about 2 s) unless attn_debug_set_wait_limit lowered it. Passed as a kernel argument.
long long wait_limit_cycles();

// Device address of the library's status word on the current device.
int status_word_ptr(unsigned **out);

// Decode work split, shared by the workspace query and the launch.
int decode_chunk_len(int B, int Hkv, int max_len);
size_t decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len);
// Most stream-kernel warps whose partials fit in `bytes` of workspace (a multiple of the block's
// warp count, at most the full grid), or for batches above the stream kernel's limit the full
// grid if the chunked kernel's partials fit; 0 if nothing fits.
int decode_warps_within(int B, int Hq, int Hkv, int D, int max_len, size_t bytes);

}  // namespace gqa
