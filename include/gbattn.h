/*
 * gbattn.h -- C ABI of libgbattn.so: fused attention forward on one GB300
 * (sm_103a), in two forms.
 *
 *  attn_fwd    FlashAttention-style prefill, MHA or GQA, optional causal mask,
 *              causal sliding window and symmetric local window.
 *  mla_decode  FlashMLA-style decode: one query token per sequence, H query
 *              heads sharing one latent KV head (d_c = 512) plus a RoPE key
 *              part (d_r = 64); the values are the latent KV rows themselves.
 *
 * Both compute O = softmax(scale * Q K^T + mask) V with an online softmax, so
 * the score matrix never leaves the chip ("TileLang 学习笔记", section
 * "FlashAttention 的实现": S = Q K^T, P = softmax(S), O = P V, and the
 * running max / running sum update of "Online Softmax 的关键").  They also
 * return LSE, the natural-log log-sum-exp of each row's scaled, masked
 * scores: LSE_i = ln sum_j exp(scale * q_i . k_j) over the allowed keys j.
 *
 * Conventions for every entry point
 *  - Pointers to tensors are DEVICE pointers on the current CUDA device.  The
 *    caller allocates and owns every buffer; the library never allocates,
 *    frees or keeps a reference to them past the call.
 *  - Tensors are dense, row-major, with no padding.  bf16 is IEEE bfloat16
 *    (raw 16-bit storage); LSE is fp32.  Tensor base addresses must be 16-byte
 *    aligned (TMA requirement), else GBATTN_ERR_ALIGNMENT.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous: they return once the kernels are enqueued.  Arguments are
 *    validated first; on any error nothing is enqueued and the function
 *    returns a non-zero gbattn_status, with a message in gbattn_last_error().
 *  - Every wait inside the kernels is bounded.  A wait that runs out records
 *    an error in a per-library device status word and the kernel returns
 *    without finishing; gbattn_check() reports it as GBATTN_ERR_TIMEOUT.
 *  - Thread safety: calls may come from several host threads; the last-error
 *    message is per host thread.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GBATTN_OK = 0,
    GBATTN_ERR_INVALID_ARG = 1,   /* null pointer, negative size, H % H_kv != 0, ... */
    GBATTN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d not in {64,128}) */
    GBATTN_ERR_ALIGNMENT = 3,     /* a tensor base address is not 16-byte aligned */
    GBATTN_ERR_WORKSPACE = 4,     /* workspace missing, too small or misaligned */
    GBATTN_ERR_LAUNCH = 5,        /* CUDA runtime/driver error while preparing or launching */
    GBATTN_ERR_TIMEOUT = 6,       /* a device-side bounded wait ran out (from gbattn_check) */
    GBATTN_ERR_ARCH = 7           /* current device is not compute capability 10.3 (sm_103) */
} gbattn_status;

/*
 * attn_fwd -- prefill attention forward.
 *
 * Operation ("TileLang 学习笔记", FlashAttention 的实现; the score mask is the
 * additive 0 / -inf mask of the problem statement):
 *   s_ij  = scale * sum_k Q[b,h,i,k] K[b,g,j,k]   for allowed (i, j), else -inf
 *   O[b,h,i,:] = sum_j softmax_j(s_i.) V[b,g,j,:],  LSE[b,h,i] = ln sum_j exp(s_ij)
 * with g = h / (H / H_kv) (query heads in contiguous groups share a KV head;
 * the FlashMLA article, section 5.1, shows the one-KV-head case).
 * Allowed keys, with off = N_kv - N_q (bottom-right alignment):
 *   causal = 0, window <= 0 : every key j in [0, N_kv)
 *   causal = 1              : j <= i + off
 *   causal = 1, window > 0  : i + off - window + 1 <= j <= i + off
 *   causal = 0, window > 0  : i + off - window <= j <= i + off + window
 *                             (the symmetric local window of the study notes'
 *                             local-attention variant: seqpos - w .. seqpos + w)
 * A row with no allowed key gets O = 0 and LSE = -inf.
 *
 * Arguments
 *   Q    bf16 [B, H,    N_q,  d]     K, V  bf16 [B, H_kv, N_kv, d]
 *   O    bf16 [B, H,    N_q,  d]     (written; fp32 accumulation, rounded to nearest even)
 *   LSE  fp32 [B, H,    N_q]         (written)
 *   d in {64, 128};  B, H, H_kv >= 1;  H % H_kv == 0;  N_q, N_kv >= 0;
 *   scale finite and > 0 (usually 1/sqrt(d));  causal in {0, 1};
 *   window <= 0 means no window.
 * O and LSE must not overlap the inputs.
 */
int attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
             int B, int H, int H_kv, int N_q, int N_kv, int d,
             int causal, int window, float scale, void *stream);

/*
 * attn_fwd_sparse -- attn_fwd with a block-sparse mask (the study notes'
 * block-sparse variant: attention is computed only in the blocks a
 * block-level mask selects).
 *
 * block_mask: uint8 [B, H, ceil(N_q / 128), ceil(N_kv / 128)] on the device,
 * one byte per (batch, query head, block of 128 query rows, block of 128
 * keys); a zero byte removes those keys from those rows, on top of the
 * causal / window rules of attn_fwd (whose other arguments it shares).  A row
 * left without keys gets O = 0, LSE = -inf.  Skipped blocks are neither
 * loaded nor computed.  The mask must stay unchanged until the call has run.
 * Errors as attn_fwd (a null block_mask with N_kv > 0 is
 * GBATTN_ERR_INVALID_ARG).
 */
int attn_fwd_sparse(const void *Q, const void *K, const void *V, void *O, float *LSE,
                    const unsigned char *block_mask, int B, int H, int H_kv, int N_q, int N_kv, int d,
                    int causal, int window, float scale, void *stream);

/*
 * mla_decode_workspace_bytes -- size of the scratch buffer mla_decode needs
 * for the given shape on the current device (it depends on the device's SM
 * count).  Returns 0 for an invalid shape.
 */
size_t mla_decode_workspace_bytes(int B, int H, int N_kv, int d_c);

/*
 * mla_decode -- MLA decode attention, one query token per sequence.
 *
 * Operation (the devpress.csdn.net FlashMLA article, section 2.2: the score is
 * the latent product plus the RoPE product accumulated into one score tile;
 * the values are the latent rows):
 *   s_j = scale * (Q_nope[b,h,:] . KV_latent[b,j,:] + Q_pe[b,h,:] . K_pe[b,j,:])
 *   O[b,h,:] = sum_j softmax_j(s) KV_latent[b,j,:],   LSE[b,h] = ln sum_j exp(s_j)
 *
 * Arguments
 *   Q_nope bf16 [B, H, d_c]   Q_pe bf16 [B, H, d_r]
 *   KV_latent bf16 [B, N_kv, d_c]   K_pe bf16 [B, N_kv, d_r]
 *   O bf16 [B, H, d_c] (written)    LSE fp32 [B, H] (written)
 *   d_c = 512, d_r = 64, 1 <= H <= 128 (the heads are the rows of one
 *   128-row tile, section 2.1's [block_H, dim] query tile; with H < 128 the
 *   other rows are padding that is neither read from Q nor written), B >= 1,
 *   N_kv >= 1 (same for every sequence), scale finite and > 0.
 *   workspace: device buffer of at least mla_decode_workspace_bytes(B, H,
 *   N_kv, d_c) bytes, 16-byte aligned, owned by the caller; it holds the
 *   per-split partial results and is overwritten.  Calls that share a
 *   workspace must not overlap in time.
 */
int mla_decode(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe,
               void *O, float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale,
               void *workspace, size_t workspace_bytes, void *stream);

/*
 * mla_decode_paged_workspace_bytes -- size of the scratch buffer
 * mla_decode_paged needs for B sequences of s_q query tokens on the current
 * device (it depends on the device's SM count, not on the lengths).  Returns
 * 0 for an invalid shape.
 */
size_t mla_decode_paged_workspace_bytes(int B, int s_q, int H, int d_c);

/*
 * mla_decode_paged -- MLA decode over a paged KV cache, each sequence with
 * its own length.
 *
 * Operation: mla_decode's, with the FlashMLA article's KV loop bound
 * (section 2.2, ceildiv(seqlen_kv, block_N)) taken per sequence: sequence b
 * has keys j < cache_seqlens[b], and key j is row j % 64 of page
 * block_table[b * max_pages_per_seq + j / 64] of the caches.  With s_q query
 * tokens per sequence (several new tokens at once), the tokens are the last
 * s_q positions of the sequence and attend causally: token t sees keys
 * j < cache_seqlens[b] - (s_q - 1 - t).  A row without keys gets O = 0 and
 * LSE = -inf.  The query rows of a sequence ([s_q][H], token-major) are cut
 * into 128-row tiles of whole tokens (max(1, 128 / H) tokens each): when
 * s_q * H <= 128 all of a sequence's tokens share one tile and its keys are
 * read from memory once, each row masked to its own token's keys; with
 * H = 128 every token is its own tile and reads the keys again.
 *
 * Arguments
 *   Q_nope bf16 [B, s_q, H, d_c]   Q_pe bf16 [B, s_q, H, d_r]
 *   KV_cache bf16 [num_pages, 64, d_c]   K_pe_cache bf16 [num_pages, 64, d_r]
 *   block_table int32 [B, max_pages_per_seq] (device; entries past a
 *     sequence's last page are not read)
 *   cache_seqlens int32 [B] (device; 0 <= len <= 64 * max_pages_per_seq)
 *   O bf16 [B, s_q, H, d_c] (written)    LSE fp32 [B, s_q, H] (written)
 *   page_size = 64, d_c = 512, d_r = 64, 1 <= H <= 128, B >= 1, s_q >= 1,
 *   num_pages >= 1, max_pages_per_seq >= 1, scale finite and > 0.
 *   workspace: device buffer of at least mla_decode_paged_workspace_bytes(B,
 *   s_q, H, d_c) bytes, 16-byte aligned, owned by the caller, overwritten; calls
 *   that share a workspace must not overlap in time.
 * Rows of a sequence's last page past its length may hold anything (they
 * are zeroed on chip before the P V product).  The lengths are read on the
 * device: one outside [0, 64 * max_pages_per_seq] is clamped and reported by
 * the next gbattn_check as GBATTN_ERR_INVALID_ARG.  A block-table entry
 * outside [0, num_pages) reads zeros.
 */
int mla_decode_paged(const void *Q_nope, const void *Q_pe, const void *KV_cache, const void *K_pe_cache,
                     const int *block_table, const int *cache_seqlens, void *O, float *LSE, int B, int s_q,
                     int H, int num_pages, int max_pages_per_seq, int page_size, int d_c, int d_r, float scale,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * mla_decode_noalloc -- mla_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart of this entry point; it is a
 * convenience of this library.
 *
 * Why: some callers cannot call cudaMalloc when they call this function -- a
 * serving loop whose device memory is planned up front and must not grow, a
 * caller that must not synchronise the device (allocating and freeing may),
 * or a plain C caller without an allocator of its own.  This entry point does
 * the same computation as mla_decode, with the same arguments minus the
 * workspace, and allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.  The split-KV partial results go to a scratch array built
 * into the library instead: 21,053,440 bytes, enough for every shape on GPUs
 * with up to 160 SMs, held by every GPU that loads the library until the
 * process exits.  If the current device would need more scratch than that,
 * the call returns GBATTN_ERR_WORKSPACE and enqueues nothing.
 *
 * Set-up: the first call on each device looks up the device address of the
 * scratch array, with that device current.  Make that first call before any
 * stream capture on the device.
 *
 * All calls share the one scratch array, which keeps the contents of the last
 * call; nothing in it needs to start at zero.  Calls whose kernels overlap on
 * the GPU (for example on two streams) race on the scratch and give wrong
 * results: serialise them, or use mla_decode with one workspace per stream.
 */
int mla_decode_noalloc(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe,
                       void *O, float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale,
                       void *stream);

/*
 * attn_fwd_host_device_bytes / attn_fwd_host -- attn_fwd with Q, K, V, O and
 * LSE in HOST memory (same shapes and layouts as attn_fwd; pinned memory
 * makes the copies asynchronous, pageable memory works but copies
 * synchronously).  The call copies the inputs to a caller-owned device
 * buffer, runs attn_fwd and copies O and LSE back, cut into up to 8
 * contiguous chunks of (batch, KV-head) units so that the host-to-device
 * copies, the kernels and the device-to-host copies of different chunks
 * overlap (library-owned helper streams per device, chained to `stream` by
 * events; the chunks' kernels alternate between two of them, so consecutive
 * chunks' kernels overlap too).  Asynchronous on `stream`: O and LSE are valid once `stream`
 * reaches the point of the call (e.g. after gbattn_check(stream)).
 *   device_buf: at least attn_fwd_host_device_bytes(B, H, H_kv, N_q, N_kv, d)
 *   bytes, 256-byte aligned, owned by the caller, overwritten.
 * Errors: as attn_fwd (no alignment rule for the host pointers), plus
 * GBATTN_ERR_WORKSPACE for a missing or small device buffer.  The size
 * function returns 0 for an invalid shape.
 */
size_t attn_fwd_host_device_bytes(int B, int H, int H_kv, int N_q, int N_kv, int d);
int attn_fwd_host(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int H_kv, int N_q,
                  int N_kv, int d, int causal, int window, float scale, void *device_buf, size_t device_bytes,
                  void *stream);

/*
 * mla_decode_host_device_bytes / mla_decode_host -- mla_decode with every
 * tensor in HOST memory (same shapes and layouts), pipelined the same way
 * over up to 4 chunks of sequences.  device_buf holds the device copies and
 * the split-KV workspace: at least mla_decode_host_device_bytes(B, H, N_kv,
 * d_c, d_r) bytes, 256-byte aligned, caller-owned.  Errors: as mla_decode
 * (no alignment rule for the host pointers), GBATTN_ERR_WORKSPACE for the
 * device buffer.
 */
size_t mla_decode_host_device_bytes(int B, int H, int N_kv, int d_c, int d_r);
int mla_decode_host(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe, void *O,
                    float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale, void *device_buf,
                    size_t device_bytes, void *stream);

/*
 * ssd_scan -- Mamba-2 SSD scan, the chunk-state / chunk-scan linear-attention
 * functions benchmarked in "TileLang: 面向AI系统的可组合分块编程模型" (results,
 * linear attention on H100), with the selective-scan recurrence sketched in
 * "从FlashAttention到通用内核" section 4.  Per batch b and head h (B/C group
 * g = h / (H / G)), state S [P][N] starting at zero:
 *   S_t = exp(dt_t A_h) S_{t-1} + dt_t x_t (outer) B_t
 *   y_t = S_t C_t + D_h x_t
 * computed in chunks of 128 steps on the tensor cores (the state is carried
 * between chunks on chip, fp32).  The chunk-internal weights
 * exp(cum_t - cum_s) dt_s (C_t . B_s), the decayed B rows and the carried
 * state enter the tensor-core products rounded to bf16; sums are fp32.
 *
 * Arguments
 *   x bf16 [Bsz, L, H, P]   dt fp32 [Bsz, L, H]   A fp32 [H]
 *   B, C bf16 [Bsz, L, G, N]   D fp32 [H] or NULL (no skip term)
 *   y fp32 [Bsz, L, H, P] (written)
 *   final_state fp32 [Bsz, H, P, N] (written) or NULL
 *   P = 64, N = 128, H % G == 0, 1 <= Bsz <= 65535, L >= 1.
 *   All device pointers, caller-owned; no workspace.
 * Errors: GBATTN_ERR_INVALID_ARG, _UNSUPPORTED (other P, N), _ALIGNMENT
 * (x, B, C, y, final_state 16-byte; dt, A, D 4-byte), _LAUNCH;
 * asynchronous on `stream`.
 */
int ssd_scan(const void *x, const float *dt, const float *A, const void *B, const void *C, const float *D,
             float *y, float *final_state, int Bsz, int L, int H, int P, int G, int N, void *stream);

/*
 * gbattn_check -- synchronise `stream`, then read and clear the device status
 * word of the current device.  Returns GBATTN_OK, GBATTN_ERR_TIMEOUT if a
 * kernel's bounded wait ran out since the last check, or GBATTN_ERR_LAUNCH if
 * the stream reports a CUDA error.
 */
int gbattn_check(void *stream);

/* gbattn_last_error -- message for the calling thread's last non-OK return
 * (empty string if none).  The pointer stays valid until the thread's next call. */
const char *gbattn_last_error(void);

/*
 * gbattn_set_wait_timeout_ns -- limit for every device-side wait of later
 * launches (default 2 s; clamped to [1 ms, 60 s]).  Returns the previous value.
 */
uint64_t gbattn_set_wait_timeout_ns(uint64_t ns);

/*
 * gbattn_set_fault_injection -- test hook for the bounded waits (default 0 =
 * off).  Mode 1: in later attn_fwd launches the TMA producer never loads the
 * Q tiles, so the tensor-core warp's wait for them runs out after the wait
 * limit (gbattn_set_wait_timeout_ns); every CTA then stops, frees its tensor
 * memory and exits, and gbattn_check() returns GBATTN_ERR_TIMEOUT.  Mode 2:
 * the same for ssd_scan, whose producer then loads no chunk.  Nothing faults
 * or traps; the CUDA context stays usable.  Not part of the computation (the
 * pages have no counterpart).  Returns the previous mode.
 */
int gbattn_set_fault_injection(int mode);

/*
 * gbattn_selftest_umma -- layout check of the tensor-core building blocks the
 * kernels are made of, on one 128x128x128 bf16 tile:
 *   S = A B^T   (A, B: TMA-loaded, 128-byte-swizzled, K-major shared-memory operands)
 *   O = P V     (P written to tensor memory from registers; V a TMA-loaded,
 *                128-byte-swizzled, N-major shared-memory operand)
 * A, B, P, V: bf16 [128, 128] row-major device buffers;  S, O: fp32 [128, 128].
 * Not part of the attention computation; used by the test suite.
 */
int gbattn_selftest_umma(const void *A, const void *B, const void *P, const void *V,
                         float *S, float *O, void *stream);

/*
 * gbattn_mla_trace -- latency trace of the MLA decode kernel (observability; the
 * pages have no counterpart).  Only a library built with -DGBATTN_TRACE (the
 * package's trace build) records it; the default library returns
 * GBATTN_ERR_UNSUPPORTED and writes nothing.
 *
 * In the trace build every launch of the MLA split kernel stamps, for the
 * first GBATTN_MLA_TRACE_TILES key tiles of cluster 20 (cluster 0 when fewer
 * than 21 clusters run), the device global timer (ns) at each step of a tile's
 * chain, for both CTAs of the cluster.  This call synchronises the device,
 * copies the stamps of the launches since the last call to `host` and clears
 * them.  Layout: uint64 [2 CTAs][GBATTN_MLA_TRACE_EVENTS][GBATTN_MLA_TRACE_TILES],
 * 0 = not reached; a later launch overwrites the stamps it reaches.  Events, in
 * order: load issued, S MMA issued, P V issued for unit 0 and unit 1, S read
 * from tensor memory, send buffer 0 / 1 free, copy 0 / 1 issued to the peer,
 * softmax has unit 0 / 1 (both partials), P of unit 0 / 1 written.
 *   host: caller-owned, at least GBATTN_MLA_TRACE_BYTES bytes.
 * Errors: GBATTN_ERR_UNSUPPORTED (default library), GBATTN_ERR_INVALID_ARG
 * (host NULL or bytes too small), GBATTN_ERR_LAUNCH.
 */
#define GBATTN_MLA_TRACE_EVENTS 13
#define GBATTN_MLA_TRACE_TILES 64
#define GBATTN_MLA_TRACE_BYTES (8 * 2 * GBATTN_MLA_TRACE_EVENTS * GBATTN_MLA_TRACE_TILES)
int gbattn_mla_trace(void *host, size_t bytes);

/*
 * gbattn_attn_trace -- latency trace of the prefill kernel's dense forms
 * (observability; the pages have no counterpart).  Only the trace build
 * (-DGBATTN_TRACE) records it; the default library returns
 * GBATTN_ERR_UNSUPPORTED and writes nothing.
 *
 * In the trace build every launch of attn_fwd (the two-tile form: two 128-row
 * query tiles per CTA, 128-key tiles; or the pipelined one-tile form: one
 * query tile, 64-key tiles, which stamps the Q tile 0 events only) stamps, for four CTAs
 * (blocks 0, 1, grid / 3 and 2 grid / 3) and the first GBATTN_ATTN_TRACE_TILES
 * key blocks of each, the SM cycle counter at each step of a key block's chain.
 * This call synchronises the device, copies the stamps of the launches since
 * the last call to `host` and clears them.  Layout: int64
 * [GBATTN_ATTN_TRACE_CTAS][GBATTN_ATTN_TRACE_EVENTS][GBATTN_ATTN_TRACE_TILES]
 * (cycles; tile = key block - the CTA's first key block; 0 = not reached),
 * followed by int64 [GBATTN_ATTN_TRACE_CTAS][4]: each CTA's cycle counter and
 * global timer (ns) at its start, then at its end.  Events, in order (issuer:
 * tile j's V awaited, V seen, P of Q tile 0 seen, P V of Q tile 0 issued, K of
 * tile j + 1 seen, S of Q tile 0 for tile j + 1 issued, P of Q tile 1 seen, P V
 * of Q tile 1 issued, S of Q tile 1 for tile j + 1 issued; then for each Q tile's
 * softmax warpgroup: S seen, scores loaded, row maximum, exponentials and P
 * stored, P-ready arrive).
 *   host: caller-owned, at least GBATTN_ATTN_TRACE_BYTES bytes.
 * Errors: GBATTN_ERR_UNSUPPORTED (default library), GBATTN_ERR_INVALID_ARG
 * (host NULL or bytes too small), GBATTN_ERR_LAUNCH.
 */
#define GBATTN_ATTN_TRACE_CTAS 4
#define GBATTN_ATTN_TRACE_EVENTS 19
#define GBATTN_ATTN_TRACE_TILES 132
#define GBATTN_ATTN_TRACE_BYTES \
    (8 * GBATTN_ATTN_TRACE_CTAS * (GBATTN_ATTN_TRACE_EVENTS * GBATTN_ATTN_TRACE_TILES + 4))
int gbattn_attn_trace(void *host, size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
