// mla_decode.cu -- MLA decode attention for sm_103a: one query token per
// sequence, 128 query heads sharing one latent KV head (512 dims) plus a
// 64-dim RoPE key part; the values are the latent rows.
//
// What is computed (the devpress.csdn.net FlashMLA article, section 2.2): per
// key tile, the score tile is the latent product Q_nope KV^T plus the RoPE
// product Q_pe K_pe^T accumulated into one accumulator, followed by the
// exp2-based running max / running sum update of its section 3.1 and the
// value product P KV.  The heads form the rows of the tile (section 2.1: the
// query tile is [heads, dim]).
//
// GB300 mapping.  The fp32 output accumulator of 128 heads x 512 latent dims
// fills one SM's whole tensor memory, so a pair of CTAs (a 2-CTA cluster)
// shares each work item and splits both the contraction and the output:
//   CTA r holds latent dims [256 r, 256 r + 256) and RoPE dims [32 r, 32 r + 32):
//         its Q part and key tiles cover those 288 dims; it computes the
//         partial score over them and owns O[:, 256 r : 256 r + 256).
// (The RoPE halves are 64-byte rows, loaded and read with the 64-byte swizzle.)
// Every KV byte is read from HBM by exactly one CTA.  The two fp32 partial
// score tiles are swapped in 32-key units (128 heads x 32 keys, 16 KB) with
// one bulk copy per CTA per unit (TMA engine, shared memory to the peer's
// shared memory), so both CTAs hold the same full scores and run the same
// online softmax; each then multiplies P by its own latent half
// (V = KV_latent).  Send and receive buffers, and P in TMEM, are
// double-buffered, so the copy of one unit overlaps the softmax of the other
// and the next tile's S overlaps both.
//
// Work split: the B * ceil(N_kv / 64) key tiles are cut into one contiguous
// range per cluster (as many clusters as fit on the GPU at once).  A range
// that covers a whole sequence writes the final O and LSE; a partial range
// writes O / l (bf16) and its LSE to the workspace, and a small combine
// kernel, launched as a programmatic dependent of the split kernel so that
// its blocks are already resident when the split kernel ends, merges the
// pieces of each split sequence with the exact log-sum-exp rule (TileLang
// 学习笔记, "Online Softmax 的关键", applied across key ranges).  Only the
// first and the last sequence of a cluster's range can be partial, so the
// workspace holds two slots per cluster whatever B and N_kv are.
//
// Per CTA (384 threads, one CTA per SM):
//   warps 0, 2  TMA producers (each owns alternate stages of one 4-stage ring):
//               each range's query part (two slots), then this CTA's dims of
//               its 64-key tiles;
//   warp 1      tcgen05 issuer: S_part = Q_part K_part^T per tile (Q from
//               TMEM, N = 64) and O_half += P V_half per unit (P from TMEM,
//               N = 256), each issued as soon as its inputs are ready;
//   warps 4-7   sender (one thread per head): each range's Q part from the
//               ring into TMEM (the next range's as soon as the last S of the
//               current one is read); per tile read S_part and, per unit,
//               write it to a send buffer and copy that to the peer;
//   warps 8-11  softmax (one thread per head): own + peer partial scores,
//               online softmax, P (bf16) into TMEM, O rescaling, epilogue.
// TMEM: O half [0, 256), S [256, 320), P [320, 352) (two 16-column units),
// Q part [352, 496).
#include <cmath>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "gbattn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kH = 128;                   // heads per tile (MMA M)
constexpr int kBN = 64;                   // keys per tile (TMA stage, S MMA N)
constexpr int kBU = 32;                   // keys per unit (exchange, softmax, PV)
// Trace build: events per tile, tiles per cluster and the cluster recorded.
enum TraceEvent : int {
    kTrLoad = 0, kTrSIssue, kTrPV0, kTrPV1, kTrSRead, kTrSendBuf0, kTrSendBuf1, kTrCopy0, kTrCopy1,
    kTrSoftmax0, kTrSoftmax1, kTrP0, kTrP1, kTraceEvents
};
#ifdef GBATTN_TRACE
constexpr int kTraceTiles = 64;
constexpr int kTraceCluster = 20;
#endif
constexpr int kDc = 512;
constexpr int kHalf = 256;                // latent dims owned by one CTA
constexpr int kKvChunk = kBN * 128;       // [64 keys x 64 dims] bf16, one TMA box
constexpr int kRopeBytes = kBN * 64;      // [64 keys x 32 dims] bf16: this CTA's RoPE half of a key tile
constexpr int kStageBytes = 4 * kKvChunk + kRopeBytes;   // 4 latent chunks + the RoPE half (36 KB)
constexpr int kSSteps = 18;               // 16-dim K-steps of a CTA's score part (256 latent + 32 RoPE dims)
constexpr int kStages = 4;
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;
constexpr uint32_t kColP = 320;
constexpr uint32_t kColQ = 352;
constexpr int kXBytes = kH * kBU * 4;     // one unit of partial scores (fp32, 128-byte rows)
constexpr int kQChunk = kH * 128;         // [128 heads x 64 dims] bf16, one TMA box of Q_nope
constexpr int kQpeBytes = 64 * 64;        // [64 heads x 32 dims] bf16, one TMA box of Q_pe (64-byte swizzle)
static_assert(2 * kQChunk + kQpeBytes <= kStageBytes, "a query slot fits a ring stage");
constexpr uint32_t kBarX = 1, kBarS = 2;  // named barriers of the sender / softmax warps
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;
// Split-KV partial results (O / l of a part of an entry's keys) are stored in
// bf16 (true: fp32).  fp32 partials round the merged output once instead of
// twice but double the partials' traffic: measured 13 % slower on 64
// sequences of 4096 keys, where about 150 of the partials are written and
// read back.
constexpr bool kF32Partials = false;
using PartT = std::conditional_t<kF32Partials, float, __nv_bfloat16>;

struct Ctl {
    uint64_t q_full, q_empty;
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full, s_free;
    uint64_t sent[2], own_free[2];      // this CTA's partial of a unit: written / read by the softmax
    uint64_t xfull[2], xfree[2];        // the peer's partial of a unit: arrived / read (remote arrive)
    uint64_t p_full[2], pfree[2];       // P unit buffer: written / read by its MMA
    uint64_t o_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes =
    1024 + static_cast<size_t>(kStages) * kStageBytes + 4 * static_cast<size_t>(kXBytes) + sizeof(Ctl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kStages % 2 == 0, "the two producer warps own alternate stages");

struct Params {
    __nv_bfloat16 *O;
    float *LSE;
    PartT *ws_O;        // [slots][128][512], O / l of partial ranges
    float *ws_LSE;      // [slots][128]
    int B, N_kv, ntile;
    long long T;        // B * ntile
    int C;              // clusters launched (the tiles are split over min(C, T) of them)
    // Paged form only (sequences of their own lengths, 64-key pages):
    const int *tile_start;    // [B + 1] first flat tile of each sequence; tile_start[B] = all tiles
    const int *seq_len;       // [B] keys of each sequence (clamped to the block table's capacity)
    const int *block_table;   // [sequences][max_pages] page of each 64-key tile
    int max_pages;
    // Work entries: B counts entries; an entry is up to 128 query rows of one
    // sequence that share its keys.  A sequence has s_q query tokens of H heads
    // (its query rows are [s_q][H], token-major); an entry takes tpe
    // consecutive tokens (tpe = max(1, 128 / H)), so a sequence has epb =
    // ceil(s_q / tpe) entries: entry e is group e % epb of sequence e / epb.
    int H, s_q, tpe, epb;
    int max_seg;        // workspace slots per cluster (2: its first and last range)
    float c;            // scale * log2(e)
    int *status;
    uint64_t timeout_ns;
};

// Key-tile range of cluster cl: [range_start(cl), range_start(cl + 1)).
__host__ __device__ __forceinline__ long long range_start(long long cl, long long T, int C)
{
    return cl * T / C;
}

// Entry geometry (see Params): the sequence, the first query token, the
// number of tokens and the first query row (within the sequence's s_q * H
// rows) of entry e.
struct Entry {
    int seq, t0, nt, row0;
};
template <bool kPaged = true>
__host__ __device__ __forceinline__ Entry entry_of(int e, const Params &p)
{
    Entry x;
    if constexpr (!kPaged) {      // dense form: one token of H <= 128 heads per sequence
        x.seq = e;
        x.t0 = 0;
        x.nt = 1;
        x.row0 = 0;
        return x;
    }
    x.seq = e / p.epb;
    x.t0 = (e % p.epb) * p.tpe;
    x.nt = min(p.tpe, p.s_q - x.t0);
    x.row0 = x.t0 * p.H;
    return x;
}

// The cluster whose range holds flat tile x.
__host__ __device__ __forceinline__ int cluster_of_tile(long long x, long long T, int C)
{
    return static_cast<int>(((x + 1) * C - 1) / T);
}

// Where each sequence's key tiles sit in the flat tile space: dense (every
// sequence N_kv keys, B * ntile tiles) or paged (per-sequence lengths, prefix
// sums computed on the device by mla_tiles_kernel).
template <bool kPaged>
struct SeqMap {
    const Params &p;
    // first flat tile of sequence b (b <= B)
    __device__ __forceinline__ long long start(int b) const
    {
        if constexpr (kPaged)
            return p.tile_start[b];
        else
            return static_cast<long long>(b) * p.ntile;
    }
    __device__ __forceinline__ int keys(int b) const
    {
        if constexpr (kPaged)
            return p.seq_len[b];
        else
            return p.N_kv;
    }
    // the sequence holding flat tile x (0 <= x < total()); empty sequences own no tile
    __device__ __forceinline__ int of_tile(long long x) const
    {
        if constexpr (kPaged) {
            int lo = 0, hi = p.B;      // the last b with start(b) <= x
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (p.tile_start[mid] <= x)
                    lo = mid;
                else
                    hi = mid;
            }
            return lo;
        } else {
            return static_cast<int>(x / p.ntile);
        }
    }
    __device__ __forceinline__ long long total() const
    {
        if constexpr (kPaged)
            return p.tile_start[p.B];
        else
            return p.T;
    }
};

__device__ __forceinline__ void bulk_wait_read_allow1()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// S_part = Q_part K_part^T over the 18 16-dim steps of this CTA's part: A = Q
// from TMEM (8 columns per step), B = the stage's latent chunks (K-major,
// 128-byte swizzle, 32 bytes per step) and then its RoPE half (64-byte swizzle).
__device__ __forceinline__ void issue_s(uint32_t d, uint32_t a, uint64_t kvd, uint64_t rpd, uint32_t idesc)
{
#pragma unroll
    for (int k = 0; k < 16; ++k)
        umma_ts(d, a + k * 8, desc_advance(kvd, (k / 4) * kKvChunk + (k % 4) * 32), idesc, k > 0 ? 1u : 0u);
#pragma unroll
    for (int k = 16; k < kSSteps; ++k) umma_ts(d, a + k * 8, desc_advance(rpd, (k - 16) * 32), idesc, 1u);
}

// Event stamps for latency studies, compiled in only with -DGBATTN_TRACE (the
// library's trace build): per tile of one cluster's range, the global timer (ns)
// at each step of the tile's chain, [CTA rank][event][tile], 0 = not reached.
// The events are listed with gbattn_mla_trace in the public header.
#ifdef GBATTN_TRACE
__device__ unsigned long long g_mla_trace[2][kTraceEvents][kTraceTiles];
#define MLA_TRACE(e, i)                                                                         \
    do {                                                                                        \
        if (cl == (p.C > kTraceCluster ? kTraceCluster : 0) && (i) >= 0 && (i) < kTraceTiles)   \
            g_mla_trace[rank][e][i] = global_timer_ns();                                        \
    } while (0)
#else
#define MLA_TRACE(e, i) \
    do {                \
    } while (0)
#endif

template <bool kPaged>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ CUtensorMap tmKp,
                     const __grid_constant__ CUtensorMap tmQn, const __grid_constant__ CUtensorMap tmQp, const Params p)
{
    const SeqMap<kPaged> S{p};
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sKV = smem;                                   // [stage][chunk][64 keys][128 B]
    uint8_t *sSend = sKV + kStages * kStageBytes;          // [2][128 rows][128 B] fp32, swizzled
    uint8_t *sRecv = sSend + 2 * kXBytes;                  // [2][128 rows][128 B] fp32, swizzled
    Ctl &c = *reinterpret_cast<Ctl *>(sRecv + 2 * kXBytes);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int cl = blockIdx.x / 2;
    const int dim0 = static_cast<int>(rank) * kHalf;

    if (threadIdx.x == 0) {
        mbar_init(&c.q_full, 128);
        mbar_init(&c.q_empty, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], 1);
        }
        mbar_init(&c.s_full, 1);
        mbar_init(&c.s_free, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&c.sent[i], 1);
            mbar_init(&c.own_free[i], 1);
            mbar_init(&c.xfull[i], 1);    // this CTA's expect_tx arrive + the peer's 16 KB
            mbar_init(&c.xfree[i], 1);    // remote arrive: the peer's receive buffer i is free
            mbar_init(&c.p_full[i], 128);
            mbar_init(&c.pfree[i], 1);
        }
        mbar_init(&c.o_empty, 128);
        mbar_init(&c.drain, 1);
        c.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    cluster_sync_all();            // the peer's barriers exist before any remote arrive or copy
    tc_fence_after_sync();
    const uint32_t tbase = c.tmem_base;
    const WaitCtl ctl{&c.abort, p.status, p.timeout_ns};
    // The combine kernel may be scheduled as soon as SMs free up; it waits for
    // this grid's completion before reading anything.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Paged form: this grid is a programmatic dependent of the tile-table
    // kernel; everything above overlapped it, the table is read below.
    if constexpr (kPaged) asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long T = S.total();
    // Partition over min(C, T) clusters, so that no cluster inside a split
    // sequence's span is empty; the clusters past that have no work.
    const int Ce = static_cast<int>(min(static_cast<long long>(p.C), T));
    const long long t_begin = cl < Ce ? range_start(cl, T, Ce) : T;
    const long long t_end = cl < Ce ? range_start(cl + 1, T, Ce) : T;
    // first and last sequence with tiles in this cluster's range (none when empty)
    const int b_first = t_end > t_begin ? S.of_tile(t_begin) : 0;
    const int b_last = t_end > t_begin ? S.of_tile(t_end - 1) : -1;

    if (warp == 0 || warp == 2) {
        // =================== TMA producers ===================
        // Two producer warps own alternate ring stages (kStages is even, so a
        // stage always belongs to the same warp): a thread's bulk-tensor loads
        // are served one after another, and two issuing warps double the
        // request rate.  Both walk the same slot sequence and issue their own.
        const int mine = warp == 0 ? 0 : 1;
        if (lane == 0) {
            if (mine == 0) {
                tma_prefetch_desc(&tmKV);
                tma_prefetch_desc(&tmKp);
                tma_prefetch_desc(&tmQn);
                tma_prefetch_desc(&tmQp);
            }
            bool ok = true;
            int it = 0;
            const uint32_t kvbytes = kStageBytes;
            const uint32_t qbytes = 2 * kQChunk + kQpeBytes;
            const int rope0 = static_cast<int>(rank) * 32;                  // this CTA's RoPE dims
            const int chunk0 = static_cast<int>(rank) * (kHalf / 64);     // this CTA's first latent chunk
            for (int b = b_first; b <= b_last && ok; ++b) {
                const long long P0 = S.start(b);
                const long long x0 = max(t_begin, P0), x1 = min(t_end, S.start(b + 1));
                if (x0 >= x1) continue;       // an empty sequence
                const Entry en = entry_of<kPaged>(b, p);
                const int *pages = kPaged ? p.block_table + static_cast<size_t>(en.seq) * p.max_pages : nullptr;
                // paged: the page of the next tile, loaded one tile ahead of its use
                int outer_next = kPaged ? __ldg(pages + (x0 - P0)) : en.seq;
                // This sequence's query part: two ring slots, each [128 heads x 64 dims]
                // chunks 2i and 2i + 1 of Q_nope (one request), plus heads [64i, 64i + 64)
                // of Q_pe on CTA 1.
                for (int qi = 0; qi < 2; ++qi, ++it) {
                    if ((it & 1) != mine) continue;
                    const int s = it % kStages;
                    const uint32_t round = static_cast<uint32_t>(it / kStages);
                    if (round > 0 && !(ok = mbar_wait(&c.empty[s], (round & 1u) ^ 1u, ctl))) break;
                    uint8_t *dst = sKV + s * kStageBytes;
                    mbar_arrive_expect_tx(&c.full[s], qbytes);
                    tma_load_4d(dst, &tmQn, &c.full[s], 0, en.row0, chunk0 + 2 * qi, en.seq);
                    tma_load_3d(dst + 2 * kQChunk, &tmQp, &c.full[s], rope0, en.row0 + qi * 64, en.seq);
                }
                for (long long x = x0; x < x1 && ok; ++x, ++it) {
                    if (mine == 0 && x == max(x0, x1 - 4) && b < b_last) {
                        // The next range's query and first key tiles into L2 a few tiles
                        // ahead: its two query slots take half the ring, so its first
                        // tile is loaded late and must not also pay the HBM latency.
                        const int nb = S.of_tile(x1);          // the next entry with tiles here
                        const Entry ne = entry_of<kPaged>(nb, p);
                        tma_prefetch_l2_4d(&tmQn, 0, ne.row0, chunk0, ne.seq);
                        tma_prefetch_l2_3d(&tmQp, rope0, ne.row0, ne.seq);
                        tma_prefetch_l2_3d(&tmQp, rope0, ne.row0 + 64, ne.seq);
                        const long long nn = min(S.start(nb + 1), t_end) - x1;
                        for (int j = 0; j < min(nn, 3LL); ++j) {
                            const int r = kPaged ? 0 : j * kBN;
                            const int o = kPaged ? __ldg(p.block_table + static_cast<size_t>(ne.seq) * p.max_pages + j)
                                                 : ne.seq;
                            tma_prefetch_l2_4d(&tmKV, 0, r, chunk0, o);
                            tma_prefetch_l2_3d(&tmKp, rope0, r, o);
                        }
                    }
                    const int tile = static_cast<int>(x - P0);          // tile of the sequence
                    // dense: rows [64 tile, 64 tile + 64) of sequence b; paged: the tile's page
                    // (read a tile ahead, so the load overlaps the slot waits)
                    const int row0 = kPaged ? 0 : tile * kBN;
                    const int outer = outer_next;
                    if (kPaged && x + 1 < x1) outer_next = __ldg(pages + tile + 1);
                    if ((it & 1) != mine) continue;
                    const int s = it % kStages;
                    const uint32_t round = static_cast<uint32_t>(it / kStages);
                    if (round > 0 && !(ok = mbar_wait(&c.empty[s], (round & 1u) ^ 1u, ctl))) break;
                    uint8_t *dst = sKV + s * kStageBytes;
                    mbar_arrive_expect_tx(&c.full[s], kvbytes);
                    MLA_TRACE(kTrLoad, static_cast<int>(x - t_begin));
                    tma_load_4d(dst, &tmKV, &c.full[s], 0, row0, chunk0, outer);   // 4 latent chunks
                    tma_load_3d(dst + 4 * kKvChunk, &tmKp, &c.full[s], rope0, row0, outer);   // RoPE half
                }
                if (!ok) break;
            }
            if (!ok) {
                // Let every load this warp issued land before the CTA exits.
                volatile int no_abort = 0;
                const WaitCtl drain{&no_abort, p.status, p.timeout_ns};
                for (int i = (it > kStages ? it - kStages : 0); i < it; ++i)
                    if ((i & 1) == mine)
                        mbar_wait(&c.full[i % kStages], static_cast<uint32_t>(i / kStages) & 1u, drain);
            }
        }
    } else if (warp == 1) {
        // =================== tensor-core issuer ===================
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kH, kBN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(kH, kHalf, false, true);
            const uint32_t sKVa = smem_u32(sKV);
            const uint32_t aFull = smem_u32(&c.full[0]), aSfree = smem_u32(&c.s_free), aQfull = smem_u32(&c.q_full);
            const uint32_t aPfull = smem_u32(&c.p_full[0]), aOempty = smem_u32(&c.o_empty);
            // Two cursors, issued as soon as their inputs are ready: S per
            // tile and PV per unit, so that S of the next tiles never waits
            // behind the softmax of an earlier unit.  Readiness is polled
            // without suspending the thread.
            const int total = static_cast<int>(t_end - t_begin);
            const long long bnd0 = S.start(b_first + 1);   // end of the first sequence's tiles
            // Ring slots: each range of the cluster starts with two query slots,
            // then one slot per key tile.
            // S cursor: tile gs (flat t_begin + gs), its ring slot and segment.
            int gs = 0, s_slot = 2, s_seg = 0;
            long long s_x = t_begin, s_bnd = bnd0;
            bool s_first = true;
            // PV cursor: unit gu of tile gu / 2.
            int gu = 0, u_slot = 2, u_seg = 0;
            long long u_x = t_begin, u_bnd = bnd0;
            bool u_first = true;
            uint64_t t_last = global_timer_ns();
            for (uint32_t spin = 1; gu < 2 * total; ++spin) {
                bool progressed = false;
                // Every barrier this pass may look at is tested at once: a test
                // whose result is branched on costs the thread ~170 cycles, and
                // tested one after another they delayed each issue by their
                // sum (a result not needed this pass is not used).
                const int ph_h = gu & 1;
                const bool r_p = mbar_poll(aPfull + ph_h * 8, static_cast<uint32_t>(gu >> 1) & 1u);
                const bool r_o = mbar_poll(aOempty, static_cast<uint32_t>(u_seg - 1) & 1u);
                const bool r_full = mbar_poll(aFull + (s_slot % kStages) * 8, static_cast<uint32_t>(s_slot / kStages) & 1u);
                const bool r_sfree = mbar_poll(aSfree, static_cast<uint32_t>(gs - 1) & 1u);
                const bool r_q = mbar_poll(aQfull, static_cast<uint32_t>(s_seg) & 1u);
                if (gu < 2 * gs) {
                    // O_half += P V_half for one unit: P from TMEM (8 columns per 16
                    // keys); V = the latent chunks of the tile's stage read N-major
                    // (64-dim blocks 8 KB apart, 16 keys = 2 KB per MMA).
                    const int h = gu & 1;
                    const bool first = h == 0 && u_first;
                    const int u_stage = u_slot % kStages;
                    if (r_p && (!first || u_seg == 0 || r_o)) {
                        tc_fence_after_sync();
                        const uint64_t vd =
                            smem_desc_sw128(sKVa + u_stage * kStageBytes + h * (kBU * 128), kKvChunk, 1024);
                        const uint32_t tp = tbase + kColP + h * (kBU / 2);
                        umma_ts(tbase + kColO, tp, vd, idPV, first ? 0u : 1u);
#pragma unroll
                        for (int k = 1; k < kBU / 16; ++k)
                            umma_ts(tbase + kColO, tp + k * 8, desc_advance(vd, k * 2048), idPV, 1u);
                        umma_commit(&c.pfree[h]);
                        MLA_TRACE(kTrPV0 + h, gu >> 1);
                        if (h == 1) {
                            umma_commit(&c.empty[u_stage]);
                            ++u_slot;
                            if (++u_x == u_bnd) {
                                u_slot += 2;
                                if (u_x < t_end) u_bnd = S.start(S.of_tile(u_x) + 1);
                                ++u_seg;
                                u_first = true;
                            } else {
                                u_first = false;
                            }
                        }
                        ++gu;
                        progressed = true;
                    }
                }
                if (gs < total) {
                    const int s_stage = s_slot % kStages;
                    if (r_full && (gs == 0 || r_sfree) && (!s_first || r_q)) {
                        tc_fence_after_sync();
                        // S_part = Q_part K_part^T: Q from TMEM (8 columns per 16 dims).
                        const uint64_t kvd = smem_desc_sw128(sKVa + s_stage * kStageBytes, 16, 1024);
                        const uint64_t rpd = smem_desc_sw64_kmajor(sKVa + s_stage * kStageBytes + 4 * kKvChunk);
                        issue_s(tbase + kColS, tbase + kColQ, kvd, rpd, idS);
                        umma_commit(&c.s_full);
                        MLA_TRACE(kTrSIssue, gs);
                        ++gs;
                        ++s_x;
                        if (s_x == s_bnd || gs == total) umma_commit(&c.q_empty);   // last tile of a range
                        ++s_slot;
                        if (s_x == s_bnd) {
                            s_slot += 2;
                            if (s_x < t_end) s_bnd = S.start(S.of_tile(s_x) + 1);
                            ++s_seg;
                            s_first = true;
                        } else {
                            s_first = false;
                        }
                        progressed = true;
                    }
                }
                if (progressed) {
                    spin = 0;
                    t_last = global_timer_ns();
                } else if ((spin & 15u) == 0) {
                    if (*ctl.abort) break;
                    if (global_timer_ns() - t_last > p.timeout_ns) {
                        raise_abort(ctl, kStatusWaitTimeout);
                        break;
                    }
                }
            }
            umma_commit(&c.drain);
            volatile int no_abort = 0;
            const WaitCtl drain{&no_abort, p.status, p.timeout_ns};
            mbar_wait(&c.drain, 0, drain);
        }
    } else if (warp >= 4 && warp < 8) {
        // =================== Q load + sender (one thread per head) ===================
        const int quad = warp - 4;
        const int row = quad * 32 + lane;
        const bool leader = threadIdx.x == 128;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t swz = static_cast<uint32_t>(row & 7);
        const uint32_t peer_recv[2] = {mapa_shared(smem_u32(sRecv), peer),
                                       mapa_shared(smem_u32(sRecv + kXBytes), peer)};
        const uint32_t peer_xfull[2] = {mapa_shared(smem_u32(&c.xfull[0]), peer),
                                        mapa_shared(smem_u32(&c.xfull[1]), peer)};
        // This CTA's part of the query rows of a range into TMEM (two bf16 per
        // column), from the range's two query slots of the ring (128-byte
        // swizzled rows); slot0 is the ring slot of the first.
        auto load_q = [&](int slot0) -> bool {
            for (int qi = 0; qi < 2; ++qi) {
                const int sl = slot0 + qi, st = sl % kStages;
                if (!barrier_and(kBarX, 128, mbar_wait(&c.full[st], static_cast<uint32_t>(sl / kStages) & 1u, ctl)))
                    return false;
                const uint8_t *src = sKV + st * kStageBytes;
#pragma unroll 1
                for (int j = 0; j < 2; ++j) {
                    const uint4 *rowp = reinterpret_cast<const uint4 *>(src + j * kQChunk + row * 128);
                    uint32_t r[32];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 v = rowp[k ^ swz];
                        r[4 * k] = v.x;
                        r[4 * k + 1] = v.y;
                        r[4 * k + 2] = v.z;
                        r[4 * k + 3] = v.w;
                    }
                    tmem_st_x32(tbase + lane_base + kColQ + (2 * qi + j) * 32, r);
                }
                if ((row >> 6) == qi) {   // warp-uniform: heads [64 qi, 64 qi + 64) of this CTA's Q_pe half
                    // 64-byte rows, 64-byte swizzle: 16-byte piece k of row rr sits at k ^ ((rr >> 1) & 3)
                    const int rr = row & 63;
                    const uint4 *rowp = reinterpret_cast<const uint4 *>(src + 2 * kQChunk + rr * 64);
                    uint32_t r[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = rowp[k ^ ((rr >> 1) & 3)];
                        r[4 * k] = v.x;
                        r[4 * k + 1] = v.y;
                        r[4 * k + 2] = v.z;
                        r[4 * k + 3] = v.w;
                    }
                    tmem_st_x16(tbase + lane_base + kColQ + 128, r);
                }
                named_barrier(kBarX, 128);          // every row read: the slot goes back to the producer
                if (leader) mbar_arrive(&c.empty[st]);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&c.q_full);
            return true;
        };
        bool ok = b_last < b_first || load_q(0);
        uint32_t t = 0;          // tiles of this CTA so far
        int seg = 0;             // non-empty sequences of this CTA so far
        for (int b = b_first; b <= b_last && ok; ++b) {
            const long long P0 = S.start(b);
            const long long x0 = max(t_begin, P0), x1 = min(t_end, S.start(b + 1));
            const int n = static_cast<int>(x1 - x0);
            if (n <= 0) continue;         // an empty sequence
            for (int i = 0; i < n && ok; ++i, ++t) {
                if (!(ok = barrier_and(kBarX, 128, mbar_wait(&c.s_full, t & 1u, ctl)))) break;
                tc_fence_after_sync();
                uint32_t sr[kBN];
                tmem_ld_x64(tbase + lane_base + kColS, sr);
                if (leader) MLA_TRACE(kTrSRead, static_cast<int>(t));
                tc_fence_before_sync();
                mbar_arrive(&c.s_free);
                if constexpr (kPaged) {
                    // The sequence ends inside this tile: the rows past its end hold
                    // whatever the page holds, and P = 0 there does not cancel a
                    // non-finite V.  Zero them (latent chunks) before the P V MMAs,
                    // which run after this CTA's softmax, which waits for the sends.
                    const int valid = S.keys(b) - static_cast<int>(x0 - P0 + i) * kBN;
                    if (valid < kBN) {
                        uint8_t *stage = sKV + ((2 * (seg + 1) + static_cast<int>(t)) % kStages) * kStageBytes;
                        const int pieces = (kBN - valid) * 8;        // 16-byte pieces per chunk
                        for (int k = threadIdx.x - 128; k < 4 * pieces; k += 128) {
                            const int ch = k / pieces, r = valid + (k % pieces) / 8, q = k % 8;
                            *reinterpret_cast<uint4 *>(stage + ch * kKvChunk + r * 128 + q * 16) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                if (i == n - 1 && b < b_last) {
                    // The range's last S is done, and with it every read of its query:
                    // load the next range's query now, so that its first S does not
                    // wait for this tile's sends.
                    if (!(ok = barrier_and(kBarX, 128, mbar_wait(&c.q_empty, seg & 1, ctl)) &&
                               load_q(2 * (seg + 1) + static_cast<int>(t) + 1)))
                        break;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // Send buffer h was last read by the copy of unit (t - 1, h)
                    // (at most the other buffer's copy may still be pending) and
                    // by this CTA's softmax.
                    // (both buffers' barriers tested together first: a wait costs
                    // ~170 cycles even on a completed phase)
                    bool got = true, xfree_seen = true;
                    if (leader && t > 0) {
                        const bool own_seen = mbar_poll(smem_u32(&c.own_free[h]), (t - 1) & 1u);
                        xfree_seen = mbar_poll(smem_u32(&c.xfree[h]), (t - 1) & 1u);
                        bulk_wait_read_allow1();
                        got = own_seen || mbar_wait(&c.own_free[h], (t - 1) & 1u, ctl);
                    }
                    if (leader) MLA_TRACE(kTrSendBuf0 + h, static_cast<int>(t));
                    if (!(ok = barrier_and(kBarX, 128, got))) break;
                    float4 *srow = reinterpret_cast<float4 *>(sSend + h * kXBytes + row * 128);
#pragma unroll
                    for (int q = 0; q < kBU / 4; ++q)
                        srow[q ^ swz] = make_float4(
                            __uint_as_float(sr[h * kBU + 4 * q]), __uint_as_float(sr[h * kBU + 4 * q + 1]),
                            __uint_as_float(sr[h * kBU + 4 * q + 2]), __uint_as_float(sr[h * kBU + 4 * q + 3]));
                    fence_proxy_async_smem();      // the copy engine reads the send buffer
                    named_barrier(kBarX, 128);
                    if (leader) {
                        // The peer's receive buffer h is free once its softmax read unit (t - 1, h).
                        if (t == 0 || xfree_seen || mbar_wait(&c.xfree[h], (t - 1) & 1u, ctl)) {
                            mbar_arrive_expect_tx(&c.xfull[h], kXBytes);   // the peer's unit (t, h)
                            bulk_copy_to_peer(peer_recv[h], sSend + h * kXBytes, kXBytes, peer_xfull[h]);
                            bulk_commit_group();
                            MLA_TRACE(kTrCopy0 + h, static_cast<int>(t));
                            mbar_arrive(&c.sent[h]);
                        }
                    }
                }
            }
            ++seg;
        }
        if (leader) bulk_wait_all();   // no copy of this CTA may still be writing to the peer
    } else if (warp >= 8) {
        // =================== softmax + epilogue (one thread per head) ===================
        const int quad = warp - 8;
        const int row = quad * 32 + lane;
        const bool leader = threadIdx.x == 256;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tO = tbase + lane_base + kColO;
        const float cexp = p.c;
        const float thr = kRescaleLog2 / cexp;
        const uint32_t swz = static_cast<uint32_t>(row & 7);
        const uint32_t peer_xfree[2] = {mapa_shared(smem_u32(&c.xfree[0]), peer),
                                        mapa_shared(smem_u32(&c.xfree[1]), peer)};
        bool ok = true;
        bool okw = true;         // this warp's waits so far (agreed on at the next barrier)
        uint32_t t = 0;
        int seg = 0;
        for (int b = b_first; b <= b_last && ok; ++b) {
            const long long P0 = S.start(b), P1 = S.start(b + 1);
            const long long x0 = max(t_begin, P0), x1 = min(t_end, P1);
            const int n = static_cast<int>(x1 - x0);
            if (n <= 0) continue;         // an empty sequence
            const int n_keys = S.keys(b);
            const Entry en = entry_of<kPaged>(b, p);
            // This row's keys: the entry's key count less one per later token of
            // the entry (token t of a sequence sees keys < len - (s_q - 1 - t));
            // rows past the entry's tokens are not written and see every key.
            const int nrows = en.nt * p.H;
            const int row_keys = row < nrows ? n_keys - (en.nt - 1 - row / p.H) : n_keys;
            const int min_keys = n_keys - (en.nt - 1);     // the entry's first token's keys (same for all rows)
            ++seg;
            float m_ref = -INFINITY, l = 0.f;
            for (int i = 0; i < n && ok; ++i, ++t) {
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    // A wait costs the thread ~170 cycles even on a completed phase:
                    // test the unit's three barriers (own partial sent, the peer's
                    // copy landed, P buffer h free) together without blocking, and
                    // wait only on those not yet complete.
                    const bool sent_seen = mbar_poll(smem_u32(&c.sent[h]), t & 1u);
                    const bool xfull_seen = mbar_poll(smem_u32(&c.xfull[h]), t & 1u);
                    const bool pfree_seen = t == 0 || mbar_poll(smem_u32(&c.pfree[h]), (t - 1) & 1u);
                    const bool got = (sent_seen || mbar_wait(&c.sent[h], t & 1u, ctl)) &&
                                     (xfull_seen || mbar_wait(&c.xfull[h], t & 1u, ctl));
                    float s[kBU];
                    const float4 *orow = reinterpret_cast<const float4 *>(sSend + h * kXBytes + row * 128);
                    const float4 *rrow = reinterpret_cast<const float4 *>(sRecv + h * kXBytes + row * 128);
#pragma unroll
                    for (int q = 0; q < kBU / 4; ++q) {
                        const float4 u = orow[q ^ swz];
                        const float4 v = rrow[q ^ swz];
                        s[4 * q] = u.x + v.x;
                        s[4 * q + 1] = u.y + v.y;
                        s[4 * q + 2] = u.z + v.z;
                        s[4 * q + 3] = u.w + v.w;
                    }
                    // all 128 rows read: the sender may reuse send buffer h and the
                    // peer may copy its next unit into receive buffer h
                    if (!(ok = barrier_and(kBarS, 128, got && okw))) break;
                    if (leader) MLA_TRACE(kTrSoftmax0 + h, static_cast<int>(t));
                    if (leader) {
                        mbar_arrive(&c.own_free[h]);
                        mbar_arrive_remote(peer_xfree[h]);
                    }

                    const int key0 = static_cast<int>(x0 + i - P0) * kBN + h * kBU;
                    if (key0 + kBU > min_keys) {            // a unit some row of the entry ends in
#pragma unroll
                        for (int k = 0; k < kBU; ++k)
                            if (key0 + k >= row_keys) s[k] = -INFINITY;
                    }
                    float mx = s[0];
#pragma unroll
                    for (int k = 1; k + 1 < kBU; k += 2) mx = max3(mx, s[k], s[k + 1]);
                    mx = fmaxf(mx, s[kBU - 1]);
                    const bool move = mx > m_ref + thr;
                    const float new_ref = move ? mx : m_ref;
                    const float alpha = move ? ex2_approx((m_ref - new_ref) * cexp) : 1.0f;
                    m_ref = new_ref;
                    const float base = (m_ref == -INFINITY) ? 0.f : m_ref * cexp;
                    // exponents and sums a pair of keys at a time (packed fp32)
                    const uint64_t c2 = f2_pack(cexp, cexp), nb2 = f2_pack(-base, -base);
                    uint64_t sum2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
                    uint32_t pk[kBU / 2];
#pragma unroll
                    for (int k = 0; k < kBU / 2; ++k) {
                        float x0, x1;
                        f2_unpack(fma_f2(f2_pack(s[2 * k], s[2 * k + 1]), c2, nb2), x0, x1);
                        const float p0 = ex2_approx(x0);
                        const float p1 = ex2_approx(x1);
                        sum2[k & 1] = add_f2(sum2[k & 1], f2_pack(p0, p1));
                        pk[k] = pack_bf16x2(p0, p1);
                    }
                    {
                        float a0, a1;
                        f2_unpack(add_f2(sum2[0], sum2[1]), a0, a1);
                        l = l * alpha + (a0 + a1);
                    }
                    // P buffer h was read by the MMA of unit (t - 1, h).
                    if (t > 0)
                        okw = __all_sync(0xffffffffu, pfree_seen || mbar_wait(&c.pfree[h], (t - 1) & 1u, ctl)) && okw;
                    // O must hold every earlier unit of this range before it is rescaled.
                    if ((i > 0 || h > 0) && __any_sync(0xffffffffu, move)) {
                        const bool prev = h == 1 ? mbar_wait(&c.pfree[0], t & 1u, ctl)
                                                 : mbar_wait(&c.pfree[1], (t - 1) & 1u, ctl);
                        okw = __all_sync(0xffffffffu, prev) && okw;
                        tc_fence_after_sync();
#pragma unroll 1
                        for (int ch = 0; ch < kHalf / 32; ++ch) {
                            uint32_t o[32];
                            tmem_ld_x32(tO + ch * 32, o);
#pragma unroll
                            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                            tmem_st_x32(tO + ch * 32, o);
                        }
                    }
                    tc_fence_after_sync();
                    tmem_st_x16(tbase + lane_base + kColP + h * (kBU / 2), pk);
                    tmem_st_wait();
                    tc_fence_before_sync();
                    if (leader) MLA_TRACE(kTrP0 + h, static_cast<int>(t));
                    mbar_arrive(&c.p_full[h]);
                }
            }
            if (!ok) break;

            // ---- epilogue of this range of sequence b (after its last PV)
            if (!(ok = barrier_and(kBarS, 128, mbar_wait(&c.pfree[1], (t - 1) & 1u, ctl) && okw))) break;
            tc_fence_after_sync();
            const bool whole = (x1 - x0 == P1 - P0);
            const float inv_l = l > 0.f ? 1.0f / l : 0.f;
            const float lse = l > 0.f ? (m_ref * cexp + __log2f(l)) * kLn2 : -INFINITY;
            const size_t slot = static_cast<size_t>(cl) * 2 + (b == b_first ? 0 : 1);
            // O / l of this range, bf16, to the final output (a whole entry)
            // or to the workspace slot (a part of a split entry).
            const size_t orow = static_cast<size_t>(en.seq) * p.s_q * p.H + en.row0 + row;
            const bool store = !whole || row < nrows;
            __nv_bfloat16 *obase = p.O + orow * kDc + dim0;
            PartT *pbase = p.ws_O + (slot * kH + row) * kDc + dim0;
#pragma unroll 1
            for (int ch = 0; ch < kHalf / 32; ++ch) {
                uint32_t o[32];
                tmem_ld_x32(tO + ch * 32, o);
                if (whole || !kF32Partials) {
                    uint4 v[4];
                    uint32_t *w = reinterpret_cast<uint32_t *>(v);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
                    uint4 *dst = whole ? reinterpret_cast<uint4 *>(obase + ch * 32)
                                       : reinterpret_cast<uint4 *>(pbase + ch * 32);
                    if (store) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) dst[k] = v[k];
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(pbase + ch * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                                             __uint_as_float(o[4 * k + 2]) * inv_l,
                                             __uint_as_float(o[4 * k + 3]) * inv_l);
                }
            }
            if (rank == 0 && store) {
                if (whole)
                    p.LSE[orow] = lse;
                else
                    p.ws_LSE[slot * kH + row] = lse;
            }
            tc_fence_before_sync();
            mbar_arrive(&c.o_empty);
        }
    }

    // ---- teardown: no MMA, TMA or bulk copy of this CTA is in flight
    // (drained above); the peer must be done with this CTA's shared memory
    // before either CTA exits.
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// Merge the parts of each split entry: LSE = ln sum_q e^{LSE_q},
// O = sum_q e^{LSE_q - LSE} (O_q / l_q).  One block per (entry, group of 16
// rows), 256 threads, 32 output dims per thread; entries written whole by the
// split kernel are skipped, and (paged form) an entry without keys gets
// O = 0, LSE = -inf.
template <bool kPaged>
__global__ void __launch_bounds__(256) mla_combine_kernel(const Params p)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the split kernel is complete
    const SeqMap<kPaged> S{p};
    const int b = blockIdx.x / 8, hg = blockIdx.x % 8;
    const int h = hg * 16 + threadIdx.x / 16;        // the entry's row
    const int d0 = (threadIdx.x % 16) * 32;
    const Entry en = entry_of<kPaged>(b, p);
    if (h >= en.nt * p.H) return;                    // not a query row of this entry
    const size_t orow = static_cast<size_t>(en.seq) * p.s_q * p.H + en.row0 + h;
    const long long T = S.total();
    const long long x0 = S.start(b), x1 = S.start(b + 1);
    if (x1 <= x0) {
        uint4 *dst = reinterpret_cast<uint4 *>(p.O + orow * kDc + d0);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(0, 0, 0, 0);
        if (threadIdx.x % 16 == 0) p.LSE[orow] = -INFINITY;
        return;
    }
    const int Ce = static_cast<int>(min(static_cast<long long>(p.C), T));   // clusters with work
    const int c0 = cluster_of_tile(x0, T, Ce);
    const int c1 = cluster_of_tile(x1 - 1, T, Ce);
    if (c0 == c1) return;
    auto slot_of = [&](int q) -> size_t {
        return static_cast<size_t>(q) * 2 + (b == S.of_tile(range_start(q, T, Ce)) ? 0 : 1);
    };
    // One part's 32 values of this thread: 4 (bf16) or 8 (fp32) 16-byte loads.
    constexpr int kVec = kF32Partials ? 8 : 4;
    auto load_part = [&](size_t sq, uint4 (&v)[kVec]) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.ws_O + (sq * kH + h) * kDc + d0);
#pragma unroll
        for (int k = 0; k < kVec; ++k) v[k] = src[k];
    };
    auto accumulate = [](float (&acc)[32], float w, const uint4 (&v)[kVec]) {
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const uint32_t u[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (kF32Partials) {
                    acc[4 * k + j] += w * __uint_as_float(u[j]);
                } else {
                    acc[8 * k + 2 * j] += w * __uint_as_float(u[j] << 16);
                    acc[8 * k + 2 * j + 1] += w * __uint_as_float(u[j] & 0xffff0000u);
                }
            }
        }
    };
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
    float lse;
    const int n = c1 - c0 + 1;
    // Up to kPre parts (the usual case: an entry spans two or three cluster
    // ranges) every load of the thread is issued at once.
    constexpr int kPre = kF32Partials ? 2 : 3;
    if (n <= kPre) {
        float lq[kPre];
        uint4 v[kPre][kVec];
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            lq[i] = -INFINITY;
            if (i < n) {
                const size_t sq = slot_of(c0 + i);
                lq[i] = p.ws_LSE[sq * kH + h];
                load_part(sq, v[i]);
            }
        }
        float mx = lq[0];
#pragma unroll
        for (int i = 1; i < kPre; ++i) mx = fmaxf(mx, lq[i]);
        float denom = 0.f;
#pragma unroll
        for (int i = 0; i < kPre; ++i)
            if (i < n) denom += expf(lq[i] - mx);
        lse = mx + logf(denom);
#pragma unroll
        for (int i = 0; i < kPre; ++i)
            if (i < n) accumulate(acc, expf(lq[i] - lse), v[i]);
    } else {
        float mx = -INFINITY;
        for (int q = c0; q <= c1; ++q) mx = fmaxf(mx, p.ws_LSE[slot_of(q) * kH + h]);
        float denom = 0.f;
        for (int q = c0; q <= c1; ++q) denom += expf(p.ws_LSE[slot_of(q) * kH + h] - mx);
        lse = mx + logf(denom);
        for (int q = c0; q <= c1; ++q) {
            const size_t sq = slot_of(q);
            uint4 v[kVec];
            load_part(sq, v);
            accumulate(acc, expf(p.ws_LSE[sq * kH + h] - lse), v);
        }
    }
    uint4 out[4];
    uint32_t *o = reinterpret_cast<uint32_t *>(out);
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = pack_bf16x2(acc[2 * k], acc[2 * k + 1]);
    uint4 *dst = reinterpret_cast<uint4 *>(p.O + orow * kDc + d0);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = out[k];
    if (threadIdx.x % 16 == 0) p.LSE[orow] = lse;
}

// Paged form: the key count of every entry b (the keys its last token sees:
// token t of a sequence sees keys < len - (s_q - 1 - t); lengths outside
// [0, capacity] are clamped and set the status word) and the exclusive prefix
// sum of their 64-key tile counts, tile_start[0..B].  One block.
__global__ void __launch_bounds__(1024) mla_tiles_kernel(const int *cache_seqlens, int *seq_len, int *tile_start,
                                                        Params p, int capacity)
{
    const int B = p.B, s_q = p.s_q;
    int *status = p.status;
    __shared__ int warp_sum[32];
    __shared__ int carry;
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < B; base += 1024) {
        const int b = base + threadIdx.x;
        int n = 0;
        if (b < B) {
            const Entry en = entry_of<true>(b, p);
            int len = cache_seqlens[en.seq];
            if (len < 0 || len > capacity) {
                if (en.t0 == 0) atomicCAS(status, 0, kStatusBadLength);
                len = min(max(len, 0), capacity);
            }
            len = max(len - (s_q - en.t0 - en.nt), 0);
            seq_len[b] = len;
            n = (len + kBN - 1) / kBN;
        }
        int v = n;                          // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane == 31) warp_sum[warp] = v;
        __syncthreads();
        if (warp == 0) {                    // inclusive scan of the warp totals
            int w = warp_sum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sum[lane] = w;
        }
        __syncthreads();
        const int incl = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + v;
        if (b < B) tile_start[b] = incl - n;
        __syncthreads();
        if (threadIdx.x == 1023) carry = incl;
        __syncthreads();
    }
    if (threadIdx.x == 0) tile_start[B] = carry;
}

struct Plan {
    int ntile, C, max_seg;
    long long T;
    size_t slots;
};

// Cluster count: as many 2-CTA clusters as are co-resident on the current
// device, queried once per device (the value depends on the device's SM count
// and shared memory), under a lock so that concurrent first calls agree.
int resident_clusters(int num_sms)
{
    static std::mutex mu;
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return num_sms / 2;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaFuncSetAttribute(mla_split_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemBytes)) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, mla_split_kernel<false>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    if (n <= 0) n = num_sms / 2;
    cached[dev] = n;
    return n;
}

Plan make_plan(int B, int N_kv, int clusters)
{
    Plan pl;
    pl.ntile = (N_kv + kBN - 1) / kBN;
    pl.T = static_cast<long long>(B) * pl.ntile;
    pl.C = static_cast<int>(std::min<long long>(clusters, pl.T));
    pl.max_seg = 2;
    pl.slots = static_cast<size_t>(pl.C) * pl.max_seg;
    return pl;
}

size_t plan_bytes(const Plan &pl)
{
    return pl.slots * kH * kDc * sizeof(PartT) + pl.slots * kH * sizeof(float);
}

// ---------------------------------------------------------------------------
// Built-in scratch for mla_decode_noalloc.
//
// Some callers cannot allocate device memory at call time: code running under
// a fixed device-memory plan that must not grow (a serving loop), a caller
// that must not synchronise the device (cudaMalloc and cudaFree may), or a
// plain C caller with no allocator of its own.  For them the split-KV partial
// results live in this fixed array instead of a caller-provided workspace.
// It is sized for the largest plan this kernel makes on GPUs with up to 160
// SMs: 80 two-CTA clusters x 2 partial slots x (128 x 512 bf16 O + 128 fp32
// LSE) = 21,053,440 bytes.  Every
// GPU that loads the library holds it until the process exits.
constexpr size_t kNoAllocMaxClusters = 80;
constexpr size_t kNoAllocScratchBytes =
    kNoAllocMaxClusters * 2 * (static_cast<size_t>(kH) * kDc * sizeof(PartT) + kH * sizeof(float));
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current (in host code the symbol itself is only
// a host-side stand-in, not a device address).
static void *noalloc_scratch_ptr(std::string &err)
{
    static std::mutex mu;
    static void *ptrs[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        err = std::string("mla_decode_noalloc: cudaGetDevice: ") + cudaGetErrorString(e);
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            err = std::string("mla_decode_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e);
            return nullptr;
        }
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

int launch_mla_decode_noalloc(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe,
                              void *O, float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale,
                              const LaunchEnv &env, std::string &err)
{
    void *scratch = noalloc_scratch_ptr(err);
    if (!scratch) return 5;
    const size_t need = plan_bytes(make_plan(B, N_kv, resident_clusters(env.num_sms)));
    if (need > kNoAllocScratchBytes) {
        char buf[220];
        snprintf(buf, sizeof buf,
                 "mla_decode_noalloc: this device needs %zu bytes of split-KV scratch, more than the "
                 "built-in maximum of %zu bytes; use mla_decode with a workspace",
                 need, kNoAllocScratchBytes);
        err = buf;
        return 4;
    }
    return launch_mla_decode(Q_nope, Q_pe, KV_latent, K_pe, O, LSE, B, H, N_kv, d_c, d_r, scale, scratch,
                             kNoAllocScratchBytes, env, err);
}

// Tokens of one sequence that share a 128-row entry (1 when H = 128).
static int tokens_per_entry(int H)
{
    return std::max(1, kH / H);
}

size_t mla_workspace_bytes(int B, int H, int N_kv, int d_c, int num_sms)
{
    if (B < 1 || H < 1 || H > kH || N_kv < 1 || d_c != kDc) return 0;
    return plan_bytes(make_plan(B, N_kv, resident_clusters(num_sms)));
}

int launch_mla_decode(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe, void *O,
                      float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale, void *workspace,
                      size_t workspace_bytes, const LaunchEnv &env, std::string &err)
{
    const Plan pl = make_plan(B, N_kv, resident_clusters(env.num_sms));
    if (workspace_bytes < plan_bytes(pl)) {
        err = "mla_decode: workspace too small";
        return 4;
    }
    CUtensorMap tkv, tkp, tqn, tqp;
    if (!make_tma_bf16_chunked(tkv, KV_latent, d_c, N_kv, B, kBN, 4, err) ||
        !make_tma_bf16_3d_sw64(tkp, K_pe, d_r, N_kv, B, kBN, err) ||
        !make_tma_bf16_chunked(tqn, Q_nope, d_c, H, B, kH, 2, err) ||
        !make_tma_bf16_3d_sw64(tqp, Q_pe, d_r, H, B, kH / 2, err))
        return 5;
    Params p;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.ws_O = static_cast<PartT *>(workspace);
    p.ws_LSE = reinterpret_cast<float *>(p.ws_O + pl.slots * kH * kDc);
    p.B = B;                  // one entry per sequence (one query token of H <= 128 heads)
    p.H = H;
    p.s_q = 1;
    p.tpe = tokens_per_entry(H);
    p.epb = 1;
    p.N_kv = N_kv;
    p.ntile = pl.ntile;
    p.T = pl.T;
    p.C = pl.C;
    p.max_seg = pl.max_seg;
    p.c = scale * 1.4426950408889634f;
    p.status = env.status;
    p.timeout_ns = env.timeout_ns;
    p.tile_start = nullptr;
    p.seq_len = nullptr;
    p.block_table = nullptr;
    p.max_pages = 0;
    cudaError_t e = cudaFuncSetAttribute(mla_split_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e == cudaSuccess) {
        mla_split_kernel<false><<<2 * pl.C, kThreads, kSmemBytes, env.stream>>>(tkv, tkp, tqn, tqp, p);
        e = cudaGetLastError();
    }
    bool split = false;   // does a cluster range boundary fall inside a sequence?
    for (int cl = 1; cl < pl.C && !split; ++cl) split = range_start(cl, pl.T, pl.C) % pl.ntile != 0;
    if (e == cudaSuccess && split) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(B) * 8, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = env.stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, mla_combine_kernel<false>, p);
    }
    if (e != cudaSuccess) {
        err = std::string("mla_decode launch: ") + cudaGetErrorString(e);
        return 5;
    }
    return 0;
}

// ---------------------------------------------------------------- paged form
// Workspace: split partials as in the dense form (2 slots per cluster), then
// tile_start [E + 1] and seq_len [E] (int32) for the E entries.
static size_t paged_bytes(int B, int clusters, size_t &off_tiles)
{
    const size_t slots = static_cast<size_t>(clusters) * 2;
    off_tiles = slots * kH * kDc * sizeof(PartT) + slots * kH * sizeof(float);
    return off_tiles + (2 * static_cast<size_t>(B) + 1) * sizeof(int);
}

// Entries of B sequences of s_q tokens of H heads.
static long long paged_entries(int B, int s_q, int H)
{
    const int tpe = tokens_per_entry(H);
    return static_cast<long long>(B) * ((s_q + tpe - 1) / tpe);
}

size_t mla_paged_workspace_bytes(int B, int s_q, int H, int d_c, int num_sms)
{
    if (B < 1 || s_q < 1 || H < 1 || H > kH || d_c != kDc) return 0;
    size_t off = 0;
    return paged_bytes(static_cast<int>(paged_entries(B, s_q, H)), resident_clusters(num_sms), off);
}

int launch_mla_decode_paged(const void *Q_nope, const void *Q_pe, const void *KV_cache, const void *K_pe_cache,
                            const int *block_table, const int *cache_seqlens, void *O, float *LSE, int B_seq,
                            int s_q, int H, int num_pages, int max_pages, int d_c, int d_r, float scale,
                            void *workspace, size_t workspace_bytes, const LaunchEnv &env, std::string &err)
{
    const int tpe = tokens_per_entry(H);
    const int epb = (s_q + tpe - 1) / tpe;
    const int B = static_cast<int>(paged_entries(B_seq, s_q, H));   // entries
    const int C = resident_clusters(env.num_sms);
    size_t off_tiles = 0;
    if (workspace_bytes < paged_bytes(B, C, off_tiles)) {
        err = "mla_decode_paged: workspace too small";
        return 4;
    }
    CUtensorMap tkv, tkp, tqn, tqp;
    if (!make_tma_bf16_chunked(tkv, KV_cache, d_c, kBN, num_pages, kBN, 4, err) ||
        !make_tma_bf16_3d_sw64(tkp, K_pe_cache, d_r, kBN, num_pages, kBN, err) ||
        !make_tma_bf16_chunked(tqn, Q_nope, d_c, static_cast<uint64_t>(s_q) * H, B_seq, kH, 2, err) ||
        !make_tma_bf16_3d_sw64(tqp, Q_pe, d_r, static_cast<uint64_t>(s_q) * H, B_seq, kH / 2, err))
        return 5;
    const size_t slots = static_cast<size_t>(C) * 2;
    Params p;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.ws_O = static_cast<PartT *>(workspace);
    p.ws_LSE = reinterpret_cast<float *>(p.ws_O + slots * kH * kDc);
    int *tile_start = reinterpret_cast<int *>(static_cast<char *>(workspace) + off_tiles);
    int *seq_len = tile_start + B + 1;
    p.B = B;
    p.N_kv = 0;
    p.ntile = 0;
    p.T = 0;
    p.C = C;
    p.max_seg = 2;
    p.c = scale * 1.4426950408889634f;
    p.status = env.status;
    p.timeout_ns = env.timeout_ns;
    p.tile_start = tile_start;
    p.seq_len = seq_len;
    p.block_table = block_table;
    p.max_pages = max_pages;
    p.H = H;
    p.s_q = s_q;
    p.tpe = tpe;
    p.epb = epb;
    mla_tiles_kernel<<<1, 1024, 0, env.stream>>>(cache_seqlens, seq_len, tile_start, p, max_pages * kBN);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mla_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemBytes));
    if (e == cudaSuccess) {
        // a programmatic dependent of the tile-table kernel (it waits for it
        // before reading the table)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * C, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = env.stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, mla_split_kernel<true>, tkv, tkp, tqn, tqp, p);
    }
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(B) * 8, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = env.stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, mla_combine_kernel<true>, p);
    }
    if (e != cudaSuccess) {
        err = std::string("mla_decode_paged launch: ") + cudaGetErrorString(e);
        return 5;
    }
    return 0;
}

int mla_trace_fetch(void *host, size_t bytes, std::string &err)
{
#ifdef GBATTN_TRACE
    static_assert(kTraceEvents == GBATTN_MLA_TRACE_EVENTS && kTraceTiles == GBATTN_MLA_TRACE_TILES,
                  "trace layout of the public header");
    constexpr size_t need = sizeof(g_mla_trace);
    if (host == nullptr || bytes < need) {
        err = "gbattn_mla_trace: host buffer missing or smaller than GBATTN_MLA_TRACE_BYTES";
        return GBATTN_ERR_INVALID_ARG;
    }
    void *dev = nullptr;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(host, g_mla_trace, need);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&dev, g_mla_trace);
    if (e == cudaSuccess) e = cudaMemset(dev, 0, need);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        err = std::string("gbattn_mla_trace: ") + cudaGetErrorString(e);
        return GBATTN_ERR_LAUNCH;
    }
    return GBATTN_OK;
#else
    (void)host;
    (void)bytes;
    err = "gbattn_mla_trace: this library was built without GBATTN_TRACE";
    return GBATTN_ERR_UNSUPPORTED;
#endif
}

}  // namespace gbattn
