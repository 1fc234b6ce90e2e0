// kernels.h -- host-side declarations shared by the C-ABI layer and the
// kernel translation units of libgbattn.so.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <string>

#include <cuda.h>
#include <cuda_runtime.h>

namespace gbattn {

// Device status word codes (first error wins; read and cleared by gbattn_check).
enum : int {
    kStatusOk = 0,
    kStatusWaitTimeout = 1,
    kStatusBadLength = 2,     // a per-sequence length outside [0, capacity] (clamped)
};

// Raises a kernel's dynamic shared-memory limit to `bytes` once per device
// (the attribute is per device); `done` holds one bit per device ordinal and
// may be shared by concurrent callers.
inline cudaError_t set_smem_limit_once(const void *func, size_t bytes, std::atomic<uint64_t> &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

struct LaunchEnv {
    cudaStream_t stream;
    int *status;          // device status word of the current device
    uint64_t timeout_ns;  // limit of every device-side wait
    int num_sms;          // SM count of the current device
    int inject;           // failure-injection mode for tests (0 = off)
};

// Prefill attention forward (attn_fwd).  Pointers are device pointers, already
// validated by the caller; returns a gbattn_status value.
// block_mask: nullptr, or the block-sparse mask of attn_fwd_sparse (device).
int launch_attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                    int H_kv, int N_q, int N_kv, int d, int causal, int window, float scale,
                    const uint8_t *block_mask, const LaunchEnv &env, std::string &err);

// MLA decode (mla_decode).
size_t mla_workspace_bytes(int B, int H, int N_kv, int d_c, int num_sms);
int launch_mla_decode(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe,
                      void *O, float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale,
                      void *workspace, size_t workspace_bytes, const LaunchEnv &env,
                      std::string &err);

// MLA decode over a paged KV cache with per-sequence lengths (mla_decode_paged).
size_t mla_paged_workspace_bytes(int B, int s_q, int H, int d_c, int num_sms);
int launch_mla_decode_paged(const void *Q_nope, const void *Q_pe, const void *KV_cache, const void *K_pe_cache,
                            const int *block_table, const int *cache_seqlens, void *O, float *LSE, int B, int s_q,
                            int H, int num_pages, int max_pages, int d_c, int d_r, float scale, void *workspace,
                            size_t workspace_bytes, const LaunchEnv &env, std::string &err);

// MLA decode through the library's built-in scratch instead of a workspace
// (mla_decode_noalloc); allocates nothing.
int launch_mla_decode_noalloc(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe,
                              void *O, float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale,
                              const LaunchEnv &env, std::string &err);

// MLA decode latency trace (gbattn_mla_trace): copies and clears the stamps of
// the trace build; returns a gbattn_status value (UNSUPPORTED otherwise).
int mla_trace_fetch(void *host, size_t bytes, std::string &err);

// Prefill latency trace (gbattn_attn_trace): copies and clears the two-tile
// form's stamps of the trace build; returns a gbattn_status value
// (UNSUPPORTED otherwise).
int attn_trace_fetch(void *host, size_t bytes, std::string &err);

// Mamba-2 SSD scan (ssd_scan).
int launch_ssd_scan(const void *x, const float *dt, const float *A, const void *Bm, const void *Cm, const float *D,
                    float *y, float *S_final, int Bsz, int L, int H, int P, int G, int N, const LaunchEnv &env,
                    std::string &err);

// Tensor-core layout self test (gbattn_selftest_umma).
int launch_selftest_umma(const void *A, const void *B, const void *P, const void *V, float *S,
                         float *O, const LaunchEnv &env, std::string &err);

// Build a 128-byte-swizzled bf16 TMA descriptor for a row-major tensor viewed
// as [outer][rows][cols] (cols contiguous, cols % 8 == 0), with a box of 64
// columns x box_rows rows x 1.  Out-of-range box elements read as zero.
// Returns false and fills err on failure.
bool make_tma_bf16_3d(CUtensorMap &desc, const void *base, uint64_t cols, uint64_t rows,
                      uint64_t outer, uint32_t box_rows, std::string &err);
// As make_tma_bf16_3d with boxes of 32 columns (64 bytes) x box_rows rows and
// the 64-byte swizzle (for operands split into 32-dim halves).
bool make_tma_bf16_3d_sw64(CUtensorMap &desc, const void *base, uint64_t cols, uint64_t rows, uint64_t outer,
                           uint32_t box_rows, std::string &err);
// The same row-major bf16 tensor [outer][rows][cols] (cols % 64 == 0) viewed
// as 4-D (64 columns, rows, cols / 64, outer) with a box of 64 columns x
// box_rows rows x box_chunks 64-column chunks: one load brings box_chunks
// 128-byte-swizzled [box_rows][64] blocks, stored one after another in
// shared memory ([chunk][row][64]), i.e. several 64-column boxes in one TMA
// request.
bool make_tma_bf16_chunked(CUtensorMap &desc, const void *base, uint64_t cols, uint64_t rows, uint64_t outer,
                           uint32_t box_rows, uint32_t box_chunks, std::string &err);
// 4-D bf16 (f32 = false) or fp32 tensor map, 128-byte swizzle; dims innermost
// first, strides in bytes of dims 1..3, box in elements (inner box 128 bytes).
bool make_tma_4d(CUtensorMap &desc, bool f32, const void *base, const uint64_t (&dims)[4],
                 const uint64_t (&strides)[3], const uint32_t (&box)[4], std::string &err);

// 5-D bf16 tensor map, 128-byte swizzle; dims innermost first, strides in
// bytes of dims 1..4 (any order of sizes), box in elements.
bool make_tma_5d(CUtensorMap &desc, const void *base, const uint64_t (&dims)[5], const uint64_t (&strides)[4],
                 const uint32_t (&box)[5], std::string &err);

}  // namespace gbattn
