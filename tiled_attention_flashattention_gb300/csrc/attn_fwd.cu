// attn_fwd.cu -- fused attention forward (prefill), MHA/GQA, causal, causal
// sliding window and symmetric local window, for sm_103a.
//
// What is computed (TileLang 学习笔记, "FlashAttention 的实现" and its online
// softmax formulas): for each query row, S = Q K^T over 128-key tiles, a
// running row maximum m and running sum l, P = exp(S - m), and O accumulated
// as O * exp(m_prev - m_new) + P V; at the end O / l.  The exponentials are
// base 2 with scale * log2(e) folded into one multiply-add, as in the FlashMLA
// article's section 3.1 (exp2(acc * scale - max * scale)).
//
// How it maps to the GB300 SM, two-Q-tile form (one CTA per SM, 384 threads):
//   warp 0       TMA producer: two Q tiles (2 x 128 rows) once, then K_j and
//                V_j tiles into a ring of shared-memory slots (128-byte swizzle);
//                its thread issues the Q tiles and the first K tile right after
//                initialising the barriers, before the block's setup sync, and
//                (kPf) prefetches into L2 the Q tiles of the block that will
//                take this CTA's place on the SM;
//   warp 1       tensor-core issuer: S_t = Q_t K_j^T into TMEM, then
//                O_t += P_t V_j with P_t read from TMEM (it overwrites S_t);
//   warps 4-7    softmax of Q tile 0 (one thread per row, TMEM lane = row);
//   warps 8-11   softmax of Q tile 1;
//   warps 2-3    idle.
// The two Q tiles ping-pong: while the softmax warps work on tile 0's scores,
// the tensor core computes tile 1's scores and PV products, and vice versa
// (FlashAttention-2's point about keeping non-matmul work off the critical
// path, TileLang 学习笔记 "FlashAttention-2 的改进").  The one-Q-tile forms
// (256 threads, warps 0-7) run two CTAs per SM instead, so the other CTA fills
// the tensor core while one CTA's softmax works; the dense one ("pipelined")
// works on 64-key tiles with two S buffers, issuing the score MMA of key tile
// j + 1 before the P V of tile j, so within the CTA too the next scores are
// computed while the softmax works on the current ones (see Cfg).
//
// TMEM (32-bit columns x 128 lanes): two-tile form S0 [0,128), S1 [128,256),
// O0 [256, 256+D), O1 [256+D, 256+2D); block-sparse one-tile form S [0,128),
// O [128, 128+D); pipelined form S buffers [0,64), [64,128), O [128, 128+D).
// P (bf16 pairs) overwrites the first half of its S.
//
// The running maximum is updated lazily: the reference maximum m_ref moves
// only when a new score exceeds it by more than 8 in log2 units.  Until then
// the exponentials use the stale m_ref (values up to 2^8), which is exact in
// the end because O and l are divided by the same l built with the same
// m_ref; it avoids rescaling O (a TMEM round trip) on almost every tile.
#include <algorithm>
#include <cmath>

#include "gbattn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kBM = 128;       // query rows per Q tile
constexpr int kBN = 128;       // keys per K/V tile of the two-tile and block-sparse forms (and of the mask)
constexpr int kQChunkBytes = kBM * 128;  // one TMA box of a Q (or O) tile: 128 rows x 64 bf16 (128 B)
constexpr float kRescaleLog2 = 8.0f;     // lazy-rescale threshold (log2 units)
constexpr float kLn2 = 0.693147180559945309f;

// Forms, by the number kT of 128-row Q tiles per CTA and the key tile BN:
//   kT = 2, BN = 128: one CTA per SM, 384 threads (two softmax warpgroups
//           ping-pong on the tensor core), 512 TMEM columns, a ring of 5
//           (d=128) / 10 (d=64) K/V slots;
//   kT = 1: two CTAs per SM, 256 threads (one softmax warpgroup; the other
//           CTA fills the tensor core while it works), 256 TMEM columns.  One
//           CTA's start-up and drain overlap the other's main loop, and the
//           finer work items balance better.  BN = 64 (dense, pipelined): two
//           S buffers, a ring of 4 / 10 slots of 64-key K or V tiles loaded in
//           the issuer's order (K of tile j + 1 before V of tile j); BN = 128
//           (block-sparse, whose mask is in 128-key blocks): one S, a ring of
//           2 / 5 slots.
// Registers per thread after the per-role split (setmaxnreg): warpgroup 0
// (producer, MMA issuer, idle warps) gives registers to the softmax
// warpgroups, which hold a 128-float score row per thread.  kT = 2:
// 128 * 104 + 256 * 200 = 64,512 = 384 * 168; kT = 1: 128 * 64 + 128 * 192
// (or 56 + 200 where that avoids spills; the pipelined forms, whose row is 64
// floats, 88 + 168) = 32,768 = 256 * 128, the registers each block is launched
// with.
// BN keys per K/V tile: 128, or 64 for the pipelined one-tile form (kT = 1,
// kPipe): its two 64-column S buffers let the score MMA of key tile j + 1 run
// while the softmax works on tile j, inside one CTA, and two such CTAs still
// fit an SM (256 TMEM columns, under 100 KB of shared memory each).
template <int D, int kT, int BN = kBN>
struct Cfg {
    static constexpr bool kPipe = kT == 1 && BN == 64;
    static constexpr int kChunks = D / 64;
    static constexpr int kQTileBytes = kBM * D * 2;
    static constexpr int kKvTileBytes = BN * D * 2;
    static constexpr int kKvChunkBytes = BN * 128;   // one TMA box of a K/V tile: BN rows x 64 bf16
    static constexpr int kSlots = kT == 2 ? ((D == 128) ? 5 : 10)
                                          : (kPipe ? ((D == 128) ? 4 : 10) : ((D == 128) ? 2 : 5));
    static constexpr uint32_t kTmemCols = kT == 2 ? 512 : 256;
    static constexpr int kThreads = kT == 2 ? 384 : 256;
    static constexpr int kMinBlocks = kT == 2 ? 1 : 2;
    // TMEM columns of S buffer i (P overwrites its first BN / 2) and of O_t:
    // two-tile form S_t of Q tile t at 128 t; pipelined form S buffers at 0, 64.
    __host__ __device__ static constexpr uint32_t col_s(int i) { return static_cast<uint32_t>(BN) * i; }
    __host__ __device__ static constexpr uint32_t col_o(int t) { return (kPipe ? 128u : 128u * kT) + D * t; }
};

struct Ctl {
    uint64_t q_full;
    uint64_t full[10];
    uint64_t empty[10];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_final[2];
    uint64_t pv_done;       // pipelined form: P V of a key tile complete (O stable for a rescale)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int sp_lo[2], sp_hi[2];     // block-sparse form: first / last + 1 active key block of each Q tile
};

template <int D, int kT, int BN>
constexpr size_t smem_bytes()
{
    using C = Cfg<D, kT, BN>;
    return 1024 + static_cast<size_t>(kT) * C::kQTileBytes + static_cast<size_t>(C::kSlots) * C::kKvTileBytes +
           sizeof(Ctl);
}

struct Params {
    __nv_bfloat16 *O;
    float *LSE;
    int B, H, H_kv, N_q, N_kv;
    // Visible keys of query row i, with i' = i + N_kv - N_q:
    // i' - lo_pad <= j <= i' + hi_pad (and j < N_kv); kNoPad means unbounded.
    int lo_pad, hi_pad;
    int group;          // H / H_kv
    int n_qblk;         // ceil(N_q / (128 kT))
    // Block-sparse form only: a byte per (b, h, 128-row query block, 128-key
    // block), [B][H][ceil(N_q/128)][ceil(N_kv/128)]; 0 skips the block.
    const uint8_t *block_mask;
    int mask_qb, mask_kb;
    float c;            // scale * log2(e)
    int inject;         // 1: the producer never loads the Q tiles (tests the bounded waits)
    int pf_stride;      // > 0: prefetch into L2 the Q tiles of block blockIdx.x + pf_stride
    int *status;
    uint64_t timeout_ns;
};

struct Range {
    int lo, hi;         // KV tiles [lo, hi); empty when lo >= hi
};

// Event stamps for latency studies of the dense forms (two-tile and pipelined
// one-tile), compiled in only with -DGBATTN_TRACE (the library's trace build):
// for four CTAs of a launch (blocks 0, 1, grid / 3 and 2 grid / 3) the SM cycle
// counter at each step of every key tile's chain, [CTA][event][tile], tile =
// key block - the CTA's first block, 0 = not reached; plus each CTA's cycle
// counter and global timer (ns) at its start and end, which convert cycles to
// time.  The events are listed with gbattn_attn_trace in the public header (the
// pipelined form has one Q tile: it stamps the tile-0 events only).
enum AttnTraceEvent : int {
    kAtWaitV = 0, kAtVSeen, kAtP0Seen, kAtPV0Issued, kAtKNextSeen, kAtS0NextIssued, kAtP1Seen, kAtPV1Issued,
    kAtS1NextIssued, kAtS0Seen, kAtS0Loaded, kAtMax0, kAtExp0, kAtP0Arrive, kAtS1Seen, kAtS1Loaded, kAtMax1,
    kAtExp1, kAtP1Arrive, kAtEvents
};
#ifdef GBATTN_TRACE
constexpr int kAtCtas = 4;
constexpr int kAtTiles = 132;
__device__ long long g_attn_trace[kAtCtas][kAtEvents][kAtTiles];
__device__ long long g_attn_trace_clock[kAtCtas][4];   // cycles, ns at the CTA's start; cycles, ns at its end
__device__ __forceinline__ int attn_trace_slot()
{
    const unsigned g = gridDim.x, bx = blockIdx.x;
    return bx == 0 ? 0 : bx == 1 ? 1 : bx == g / 3 ? 2 : bx == 2 * g / 3 ? 3 : -1;
}
#define ATTN_TRACE(e, i)                                                                 \
    do {                                                                                 \
        if constexpr (!kSparse) {                                                        \
            const int s_ = attn_trace_slot();                                            \
            if (s_ >= 0 && static_cast<unsigned>(i) < static_cast<unsigned>(kAtTiles))   \
                g_attn_trace[s_][e][i] = clock64();                                      \
        }                                                                                \
    } while (0)
#define ATTN_TRACE_CLOCK(k)                                                              \
    do {                                                                                 \
        if constexpr (!kSparse) {                                                        \
            const int s_ = attn_trace_slot();                                            \
            if (s_ >= 0) {                                                               \
                g_attn_trace_clock[s_][2 * (k)] = clock64();                             \
                g_attn_trace_clock[s_][2 * (k) + 1] = static_cast<long long>(global_timer_ns()); \
            }                                                                            \
        }                                                                                \
    } while (0)
#else
#define ATTN_TRACE(e, i) \
    do {                 \
    } while (0)
#define ATTN_TRACE_CLOCK(k) \
    do {                    \
    } while (0)
#endif

// BN-key tiles touched by query rows [r0, r1) (r1 > r0).
template <int BN>
__device__ __forceinline__ Range kv_range(int r0, int r1, const Params &p)
{
    const long long off = static_cast<long long>(p.N_kv) - p.N_q;
    const long long key_lo = max(0LL, r0 + off - p.lo_pad);                                   // inclusive
    const long long key_hi = min(static_cast<long long>(p.N_kv), r1 - 1 + off + p.hi_pad + 1);  // exclusive
    if (key_hi <= key_lo) return {0, 0};
    return {static_cast<int>(key_lo / BN), static_cast<int>((key_hi + BN - 1) / BN)};
}

// kPf: the CTA prefetches into L2 the Q tiles of the block that will take its
// place on the SM (compiled in only where it is used: in the two-tile form the
// extra producer code alone, never executed, cost the 16k causal MHA shape 0.3 %).
template <int D, bool kSparse, int kT, int BN, bool kPf = (kT == 1)>
__global__ void __launch_bounds__(Cfg<D, kT, BN>::kThreads, Cfg<D, kT, BN>::kMinBlocks)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const Params p)
{
    using C = Cfg<D, kT, BN>;
    constexpr bool kPipe = C::kPipe;
    static_assert(kT == 1 || BN == kBN, "the two-tile form uses 128-key tiles");
    constexpr bool kWideSoftmax = kT == 2 || (kSparse && D == 128 && !kPipe);
    // (the pipelined form's softmax holds a 64-float row: more go to the issuer)
    constexpr uint32_t kRegsLow = kT == 2 ? 104 : (kWideSoftmax ? 56 : (C::kPipe ? 88 : 64));
    constexpr uint32_t kRegsHigh = kWideSoftmax ? 200 : (C::kPipe ? 168 : 192);
    static_assert(kT == 2 ? 128 * kRegsLow + 256 * kRegsHigh <= 384 * 168
                          : 128 * kRegsLow + 128 * kRegsHigh == 256 * 128, "register split");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem;                                    // [kT][QTileBytes]
    uint8_t *ring = smem + kT * C::kQTileBytes;            // [Slots][KvTileBytes]
    Ctl &c = *reinterpret_cast<Ctl *>(ring + C::kSlots * C::kKvTileBytes);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (threadIdx.x == 0) ATTN_TRACE_CLOCK(0);

    // ---- work item: (batch, head, 128 kT-row query block), longest first
    const int nbh = p.B * p.H;
    const int bh = blockIdx.x % nbh;
    const int qb = p.n_qblk - 1 - static_cast<int>(blockIdx.x / nbh);
    const int b = bh / p.H, h = bh % p.H;
    const int kvh = b * p.H_kv + h / p.group;
    int r0[2], r1[2];
    Range rng[2];
    bool has[2];
    int lo = 0x7fffffff, hi = -1;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        r0[t] = t < kT ? qb * (kT * kBM) + t * kBM : p.N_q;     // kT = 1: tile 1 is absent
        r1[t] = min(r0[t] + kBM, p.N_q);
        rng[t] = (r0[t] < p.N_q) ? kv_range<BN>(r0[t], r1[t], p) : Range{0, 0};
        has[t] = rng[t].lo < rng[t].hi;
        if (has[t]) {
            lo = min(lo, rng[t].lo);
            hi = max(hi, rng[t].hi);
        }
    }
    if (lo > hi) lo = hi = 0;
    // Block-sparse form: the mask row of each Q tile (its 128-row query block).
    const uint8_t *mrow[2] = {nullptr, nullptr};
    if constexpr (kSparse) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (r0[t] < p.N_q)
                mrow[t] = p.block_mask + (static_cast<size_t>(bh) * p.mask_qb + r0[t] / kBM) * p.mask_kb;
    }
    auto in_rng = [&](int t, int j) { return j >= rng[t].lo && j < rng[t].hi; };
    // does Q tile t compute key block j?
    auto act = [&](int t, int j) -> bool {
        if constexpr (kSparse)
            return in_rng(t, j) && __ldg(mrow[t] + j * BN / kBN) != 0;   // mask blocks are 128 keys
        else
            return in_rng(t, j);
    };
    // the next key block after j that some Q tile computes (hi if none)
    auto next_any = [&](int j) -> int {
        int k = j + 1;
        if constexpr (kSparse)
            while (k < hi && !act(0, k) && !act(1, k)) ++k;
        return k;
    };

    // ---- setup
    if (threadIdx.x == 0) {
        mbar_init(&c.q_full, 1);
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(&c.full[i], 1);
            mbar_init(&c.empty[i], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&c.s_full[t], 1);
            mbar_init(&c.p_full[t], 4 * 32);
            mbar_init(&c.o_final[t], 1);
        }
        mbar_init(&c.pv_done, 1);
        mbar_init(&c.drain, 1);
        c.abort = 0;
        fence_mbar_init();
        if constexpr (!kSparse) {
            // Dense forms: the Q tiles and K of the first key tile (ring item 0)
            // leave before the block-wide setup sync, from the thread that
            // initialised their barriers, which is also the TMA producer.  (The
            // block-sparse form learns its first tile from the mask scan.)
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            if (p.inject != 1 && (has[0] || has[1])) {
                mbar_arrive_expect_tx(&c.q_full, (has[0] + has[1]) * C::kQTileBytes);
                for (int t = 0; t < 2; ++t)
                    if (has[t])
                        for (int ch = 0; ch < C::kChunks; ++ch)
                            tma_load_3d(sQ + t * C::kQTileBytes + ch * kQChunkBytes, &tmQ, &c.q_full,
                                        ch * 64, r0[t], bh);
            }
            if (lo < hi) {
                mbar_arrive_expect_tx(&c.full[0], C::kKvTileBytes);
                for (int ch = 0; ch < C::kChunks; ++ch)
                    tma_load_3d(ring + ch * C::kKvChunkBytes, &tmK, &c.full[0], ch * 64, lo * BN, kvh);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(&c.tmem_base, C::kTmemCols);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    if constexpr (kSparse) {
        if (warp == 2) {
            // first and last active key block of each Q tile, one scan of the mask
            for (int t = 0; t < 2; ++t) {
                int f = 0x7fffffff, l = -1;
                for (int j = rng[t].lo + lane; j < rng[t].hi; j += 32)
                    if (__ldg(mrow[t] + j * BN / kBN)) {
                        f = min(f, j);
                        l = max(l, j);
                    }
                f = __reduce_min_sync(0xffffffffu, f);
                l = __reduce_max_sync(0xffffffffu, l);
                if (lane == 0) {
                    c.sp_lo[t] = f;
                    c.sp_hi[t] = l + 1;
                }
            }
        }
    }
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = c.tmem_base;
    const WaitCtl ctl{&c.abort, p.status, p.timeout_ns};
    int first = lo;          // the first key block some Q tile computes
    if constexpr (kSparse) {
        first = hi;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            has[t] = has[t] && c.sp_hi[t] > c.sp_lo[t];   // a tile with no active block writes O = 0
            if (has[t]) first = min(first, c.sp_lo[t]);
        }
    }

    if (warp == 0) {
        // =================== TMA producer ===================
        regs_dec<kRegsLow>();
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t qbytes = 0;
            for (int t = 0; t < 2; ++t)
                if (has[t]) qbytes += C::kQTileBytes;
            if (p.inject == 1) qbytes = 0;   // nothing ever completes q_full
            if (kSparse && qbytes) {          // (dense: issued at setup)
                mbar_arrive_expect_tx(&c.q_full, qbytes);
                for (int t = 0; t < 2; ++t)
                    if (has[t])
                        for (int ch = 0; ch < C::kChunks; ++ch)
                            tma_load_3d(sQ + t * C::kQTileBytes + ch * kQChunkBytes, &tmQ, &c.q_full,
                                        ch * 64, r0[t], bh);
            }
            bool ok = true;
            int it = (!kSparse && first < hi) ? 1 : 0;     // ring items already issued
            if constexpr (kPipe) {
                // The issuer's order over the key tiles the CTA computes (all of
                // [first, hi), or the active ones of a block mask): K of the
                // first, then for each tile the K of the next one (its S runs
                // first) and the V of this one; the last tile has no next K.
                int jk = it ? next_any(first) : first;    // tiles of the next K and the next V to load
                int jv = first;
                bool k_turn = true;
                while (jv < hi && ok) {
                    const bool kv = !(k_turn && jk < hi);
                    const int tile = kv ? jv : jk;
                    const int slot = it % C::kSlots;
                    const uint32_t round = static_cast<uint32_t>(it / C::kSlots);
                    if (round > 0 && !(ok = mbar_wait(&c.empty[slot], (round & 1u) ^ 1u, ctl))) break;
                    mbar_arrive_expect_tx(&c.full[slot], C::kKvTileBytes);
                    const CUtensorMap *m = kv ? &tmV : &tmK;
                    for (int ch = 0; ch < C::kChunks; ++ch)
                        tma_load_3d(ring + slot * C::kKvTileBytes + ch * C::kKvChunkBytes, m, &c.full[slot],
                                    ch * 64, tile * BN, kvh);
                    ++it;
                    if (kv) {
                        jv = next_any(jv);
                    } else {
                        jk = next_any(jk);
                    }
                    // K(first) alone, then K(next), V(this) pairs
                    k_turn = it == 1 ? true : !k_turn;
                }
            } else {
                int j = first;
                if (it == 1) {
                    // dense: K of the first tile is out; its V goes to item 1 (round 0)
                    mbar_arrive_expect_tx(&c.full[1], C::kKvTileBytes);
                    for (int ch = 0; ch < C::kChunks; ++ch)
                        tma_load_3d(ring + C::kKvTileBytes + ch * C::kKvChunkBytes, &tmV, &c.full[1], ch * 64,
                                    j * BN, kvh);
                    it = 2;
                    j = next_any(j);
                }
                for (; j < hi && ok; j = next_any(j)) {
                    for (int kv = 0; kv < 2; ++kv) {
                        const int slot = it % C::kSlots;
                        const uint32_t round = static_cast<uint32_t>(it / C::kSlots);
                        if (round > 0 && !(ok = mbar_wait(&c.empty[slot], (round & 1u) ^ 1u, ctl))) break;
                        mbar_arrive_expect_tx(&c.full[slot], C::kKvTileBytes);
                        const CUtensorMap *m = kv ? &tmV : &tmK;
                        for (int ch = 0; ch < C::kChunks; ++ch)
                            tma_load_3d(ring + slot * C::kKvTileBytes + ch * C::kKvChunkBytes, m, &c.full[slot],
                                        ch * 64, j * BN, kvh);
                        ++it;
                    }
                }
            }
            if (kPf && ok && p.pf_stride > 0 && blockIdx.x + p.pf_stride < gridDim.x) {
                // The block that will most likely take this CTA's place on the SM
                // (one wave of resident CTAs later): its Q tiles into L2 now, a few
                // key tiles before this CTA ends, so its start does not wait on HBM.
                const int b2 = static_cast<int>(blockIdx.x) + p.pf_stride;
                const int bh2 = b2 % nbh;
                const int qb2 = p.n_qblk - 1 - b2 / nbh;
                for (int t = 0; t < kT; ++t) {
                    const int rr = qb2 * (kT * kBM) + t * kBM;
                    if (rr < p.N_q)
                        for (int ch = 0; ch < C::kChunks; ++ch) tma_prefetch_l2_3d(&tmQ, ch * 64, rr, bh2);
                }
            }
            if (!ok) {
                // Aborted: let every load already issued land before the CTA exits.
                volatile int no_abort = 0;
                const WaitCtl drain{&no_abort, p.status, p.timeout_ns};
                if (qbytes) mbar_wait(&c.q_full, 0, drain);
                for (int i = (it > C::kSlots ? it - C::kSlots : 0); i < it; ++i)
                    mbar_wait(&c.full[i % C::kSlots], static_cast<uint32_t>(i / C::kSlots) & 1u, drain);
            }
        }
    } else if (warp == 1) {
        // =================== tensor-core issuer ===================
        regs_dec<kRegsLow>();
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, BN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, false, true);
            const uint32_t sQa = smem_u32(sQ), ringa = smem_u32(ring);
            // S_t = Q_t K^T: K-major A and B, 16 bf16 (32 B) per MMA along d.
            const uint64_t qdesc[2] = {smem_desc_sw128(sQa, 16, 1024),
                                       smem_desc_sw128(sQa + C::kQTileBytes, 16, 1024)};
            // S buffer sb = Q_t K^T (16 d per MMA; the 64-d chunks of Q and K are
            // kQChunkBytes / kKvChunkBytes apart)
            auto issue_S = [&](int t, int sb, int slot) {
                const uint64_t ad = qdesc[t];
                const uint64_t bd = smem_desc_sw128(ringa + slot * C::kKvTileBytes, 16, 1024);
                umma_ss(tbase + C::col_s(sb), ad, bd, idS, 0u);
#pragma unroll
                for (int k = 1; k < D / 16; ++k) {
                    const uint32_t qoff = (k / 4) * kQChunkBytes + (k % 4) * 32;
                    const uint32_t koff = (k / 4) * C::kKvChunkBytes + (k % 4) * 32;
                    umma_ss(tbase + C::col_s(sb), desc_advance(ad, qoff), desc_advance(bd, koff), idS, 1u);
                }
            };
            // O_t += P_t V: P from TMEM (8 columns per 16 keys), V N-major
            // (64-wide d chunks 16 KB apart, 16 keys = 2048 B per MMA).
            bool started[2] = {false, false};
            auto issue_PV = [&](int t, int sb, int slot) {
                const uint64_t bd = smem_desc_sw128(ringa + slot * C::kKvTileBytes, C::kKvChunkBytes, 1024);
                umma_ts(tbase + C::col_o(t), tbase + C::col_s(sb), bd, idPV, started[t] ? 1u : 0u);
#pragma unroll
                for (int k = 1; k < BN / 16; ++k)
                    umma_ts(tbase + C::col_o(t), tbase + C::col_s(sb) + k * 8, desc_advance(bd, k * 2048), idPV, 1u);
                started[t] = true;
            };
            bool ok = true;
            int it = 0;
            uint32_t pcount[2] = {0, 0};
            if (first < hi) ok = mbar_wait(&c.q_full, 0, ctl);
            if constexpr (kPipe) {
                // One Q tile, key tiles n = 0 .. ntile - 1.  S of tile n + 1 goes to
                // the other S buffer before P V of tile n, so it runs while the
                // softmax works on tile n; that buffer's previous P was read by P V
                // of tile n - 1, issued before it.
                auto islot = [&](int i) { return i % C::kSlots; };
                auto iphase = [&](int i) { return static_cast<uint32_t>(i / C::kSlots) & 1u; };
                // ring items in the producer's order: K(0), then K(n + 1), V(n) per tile n
                // (tiles n = the key tiles the CTA computes, in order)
                int jcur = first;
                if (ok && jcur < hi && (ok = mbar_wait(&c.full[islot(0)], iphase(0), ctl))) {
                    tc_fence_after_sync();
                    issue_S(0, 0, islot(0));
                    umma_commit(&c.s_full[0]);
                    umma_commit(&c.empty[islot(0)]);
                }
                it = 1;
                for (int n = 0; jcur < hi && ok; ++n) {
                    const int jn = next_any(jcur);
                    if (jn < hi) {
                        const int ik = it++;
                        if (!(ok = mbar_wait(&c.full[islot(ik)], iphase(ik), ctl))) break;
                        ATTN_TRACE(kAtKNextSeen, n);
                        tc_fence_after_sync();
                        issue_S(0, (n + 1) & 1, islot(ik));
                        umma_commit(&c.s_full[(n + 1) & 1]);
                        umma_commit(&c.empty[islot(ik)]);
                        ATTN_TRACE(kAtS0NextIssued, n);
                    }
                    const int iv = it++;
                    ATTN_TRACE(kAtWaitV, n);
                    // V of tile n and P of tile n (one barrier per S buffer: the softmax
                    // may already have finished tile n + 1, whose S was issued above),
                    // both tested before either is waited for
                    const bool v_seen = mbar_poll(smem_u32(&c.full[islot(iv)]), iphase(iv));
                    const bool p_seen = mbar_poll(smem_u32(&c.p_full[n & 1]), static_cast<uint32_t>(n >> 1) & 1u);
                    if (!v_seen && !(ok = mbar_wait(&c.full[islot(iv)], iphase(iv), ctl))) break;
                    ATTN_TRACE(kAtVSeen, n);
                    if (!p_seen && !(ok = mbar_wait(&c.p_full[n & 1], static_cast<uint32_t>(n >> 1) & 1u, ctl))) break;
                    ATTN_TRACE(kAtP0Seen, n);
                    tc_fence_after_sync();
                    issue_PV(0, n & 1, islot(iv));
                    ATTN_TRACE(kAtPV0Issued, n);
                    umma_commit(&c.empty[islot(iv)]);
                    umma_commit(&c.pv_done);
                    jcur = jn;
                }
            } else if (ok && first < hi) {
                const int slotK = 0;
                ok = mbar_wait(&c.full[slotK], 0, ctl);
                ++it;
                if (ok) {
                    tc_fence_after_sync();
                    for (int t = 0; t < 2; ++t)
                        if (act(t, first)) {
                            issue_S(t, t, slotK);
                            umma_commit(&c.s_full[t]);
                        }
                    umma_commit(&c.empty[slotK]);
                }
            }
            // Key blocks in the producer's order (every block some Q tile computes):
            // PV of block j for tile 0, S of the next block for tile 0, PV of j for
            // tile 1, S of the next block for tile 1.
            // K / V tiles are usually in the ring long before they are used, but a
            // wait on a phase that has already completed still costs the issuing
            // thread ~170 cycles.  Their barriers are tested without blocking
            // (mbar_poll) ahead of an MMA issue, so the test's latency hides behind
            // it, and the wait is skipped when the tile has landed (not in the
            // block-sparse form, whose issuer has no registers to spare; measured
            // slower in the pipelined one-tile form).
            bool v_seen = false;
            auto ring_poll = [&](int i) {
                return mbar_poll(smem_u32(&c.full[i % C::kSlots]), static_cast<uint32_t>(i / C::kSlots) & 1u);
            };
            for (int j = first; j < hi && ok && !kPipe;) {
                const int slotV = it % C::kSlots;
                ATTN_TRACE(kAtWaitV, j - first);
                if (!v_seen && !(ok = mbar_wait(&c.full[slotV], static_cast<uint32_t>(it / C::kSlots) & 1u, ctl)))
                    break;
                ++it;
                ATTN_TRACE(kAtVSeen, j - first);
                // (item `it` is the next block's K when there is one; otherwise the
                // test's result is not used)
                const bool k_seen = !kSparse && ring_poll(it);
                if (act(0, j)) {
                    if (!(ok = mbar_wait(&c.p_full[0], pcount[0]++ & 1u, ctl))) break;
                    ATTN_TRACE(kAtP0Seen, j - first);
                    tc_fence_after_sync();
                    issue_PV(0, 0, slotV);
                    ATTN_TRACE(kAtPV0Issued, j - first);
                }
                const int jn = next_any(j);
                int slotK = -1;
                v_seen = false;
                if (jn < hi) {
                    slotK = it % C::kSlots;
                    if (!k_seen && !(ok = mbar_wait(&c.full[slotK], static_cast<uint32_t>(it / C::kSlots) & 1u, ctl)))
                        break;
                    ++it;
                    ATTN_TRACE(kAtKNextSeen, j - first);
                    v_seen = !kSparse && ring_poll(it);
                    if (act(0, jn)) {
                        issue_S(0, 0, slotK);
                        umma_commit(&c.s_full[0]);
                        ATTN_TRACE(kAtS0NextIssued, j - first);
                    }
                }
                if (act(1, j)) {
                    if (!(ok = mbar_wait(&c.p_full[1], pcount[1]++ & 1u, ctl))) break;
                    ATTN_TRACE(kAtP1Seen, j - first);
                    tc_fence_after_sync();
                    issue_PV(1, 1, slotV);
                    ATTN_TRACE(kAtPV1Issued, j - first);
                }
                umma_commit(&c.empty[slotV]);
                if (slotK >= 0) {
                    if (act(1, jn)) {
                        issue_S(1, 1, slotK);
                        umma_commit(&c.s_full[1]);
                        ATTN_TRACE(kAtS1NextIssued, j - first);
                    }
                    umma_commit(&c.empty[slotK]);
                }
                j = jn;
            }
            for (int t = 0; t < 2; ++t)
                if (has[t]) umma_commit(&c.o_final[t]);
            // No tensor-core work may still be in flight when TMEM is freed.
            umma_commit(&c.drain);
            volatile int no_abort = 0;
            const WaitCtl drain{&no_abort, p.status, p.timeout_ns};
            mbar_wait(&c.drain, 0, drain);
        }
    } else if (warp < 4) {
        regs_dec<kRegsLow>();
    } else {
        // =================== softmax: one thread per query row ===================
        regs_inc<kRegsHigh>();
        const int t = (warp - 4) / 4;
        const int quad = warp % 4;                 // TMEM lanes [32*quad, 32*quad+32)
        const int row = r0[t] + quad * 32 + lane;
        const bool row_valid = row < p.N_q && r0[t] < p.N_q;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tO = tbase + lane_base + C::col_o(t);
        const float cexp = p.c;
        const float thr = kRescaleLog2 / cexp;     // threshold in raw score units
        const long long off = static_cast<long long>(p.N_kv) - p.N_q;
        // this row's visible keys: key_min <= key <= key_max (key_max < N_kv)
        const int key_max = static_cast<int>(min(row + off + p.hi_pad, static_cast<long long>(p.N_kv) - 1));
        const int key_min = static_cast<int>(max(row + off - p.lo_pad, -1LL));

        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        int n = 0;
        for (int j = rng[t].lo; j < rng[t].hi && ok; ++j, ++n) {
            if constexpr (kSparse) {
                if (!act(t, j)) {              // a block this tile skips (warp-uniform)
                    --n;
                    continue;
                }
            }
            // S buffer and its phase: Q tile t's own (two-tile / one-tile form), or
            // alternating between two (pipelined form; each buffer every other tile).
            const int sb = kPipe ? (n & 1) : t;
            const uint32_t sphase = static_cast<uint32_t>(kPipe ? (n >> 1) : n) & 1u;
            const uint32_t tS = tbase + lane_base + C::col_s(sb);
            // tcgen05.ld/st below are warp-collective: keep the outcome warp-uniform.
            ok = __all_sync(0xffffffffu, mbar_wait(&c.s_full[sb], sphase, ctl));
            if (!ok) break;
            if (quad == 0 && lane == 0) ATTN_TRACE(kAtS0Seen + 5 * t, j - first);
            tc_fence_after_sync();
            float s[BN];
            {
                uint32_t sr[BN];
                if constexpr (BN == 128)
                    tmem_ld_4x32(tS, sr);
                else
                    tmem_ld_x64(tS, sr);
#pragma unroll
                for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(sr[i]);
            }
            if (quad == 0 && lane == 0) ATTN_TRACE(kAtS0Loaded + 5 * t, j - first);

            const int k0 = j * BN;
            const bool need_mask = (k0 + BN > p.N_kv) || (k0 + BN - 1 > r0[t] + off + p.hi_pad) ||
                                   (k0 < (r1[t] - 1) + off - p.lo_pad);
            if (need_mask) {
                if constexpr (kPipe) {
                    // key k0 + i is visible iff 0 <= i - lo_i <= span: one unsigned
                    // compare per element (a row without keys masks everything)
                    const int span = key_max - key_min;
                    const int lo_i = span < 0 ? (1 << 30) : key_min - k0;
                    const uint32_t uspan = span < 0 ? 0u : static_cast<uint32_t>(span);
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (static_cast<uint32_t>(i - lo_i) > uspan) s[i] = -INFINITY;
                } else {
#pragma unroll
                    for (int i = 0; i < BN; ++i) {
                        const int key = k0 + i;
                        const bool allowed = key >= key_min && key <= key_max;
                        if (!allowed) s[i] = -INFINITY;
                    }
                }
            }
            // Row maximum as four independent chains and a tree, not one
            // (BN - 1)-deep dependency chain; three-input max, two elements
            // per instruction.
            float m4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                m4[q] = s[q];
                int i = 4 + q;
#pragma unroll
                for (; i + 4 < BN; i += 8) m4[q] = max3(m4[q], s[i], s[i + 4]);
                if (i < BN) m4[q] = fmaxf(m4[q], s[i]);
            }
            const float mx = max3(fmaxf(m4[0], m4[1]), m4[2], m4[3]);
            if (quad == 0 && lane == 0) ATTN_TRACE(kAtMax0 + 5 * t, j - first);

            const bool move = mx > m_ref + thr;
            const float new_ref = move ? mx : m_ref;
            const float alpha = move ? ex2_approx((m_ref - new_ref) * cexp) : 1.0f;
            m_ref = new_ref;
            const float base = (m_ref == -INFINITY) ? 0.f : m_ref * cexp;
            // Exponentials a pair of keys at a time: one packed multiply-add
            // for the two exponents, one packed add into the running sums (two
            // independent pairs of partial sums).
            const uint64_t c2 = f2_pack(cexp, cexp), nb2 = f2_pack(-base, -base);
            uint64_t sum2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    f2_unpack(fma_f2(f2_pack(s[q * 32 + 2 * i], s[q * 32 + 2 * i + 1]), c2, nb2), x0, x1);
                    const float p0 = ex2_approx(x0);
                    const float p1 = ex2_approx(x1);
                    sum2[i & 1] = add_f2(sum2[i & 1], f2_pack(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st_x16(tS + q * 16, pk);
            }
            if (quad == 0 && lane == 0) ATTN_TRACE(kAtExp0 + 5 * t, j - first);
            {
                float a0, a1;
                f2_unpack(add_f2(sum2[0], sum2[1]), a0, a1);
                l = l * alpha + (a0 + a1);
            }
            if (n > 0 && __any_sync(0xffffffffu, move)) {
                // O_t already holds the PV products of earlier tiles; rescale it
                // before this tile's PV, which waits for p_full below.  Their
                // completion is covered by this tile's S commit, except in the
                // pipelined form, where S of this tile was issued before P V of
                // the previous one: wait for that one's commit.
                if constexpr (kPipe) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&c.pv_done, static_cast<uint32_t>(n - 1) & 1u, ctl));
                    if (!ok) break;
                    tc_fence_after_sync();
                }
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld_x32(tO + ch * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_x32(tO + ch * 32, o);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            if (quad == 0 && lane == 0) ATTN_TRACE(kAtP0Arrive + 5 * t, j - first);
            mbar_arrive(&c.p_full[sb]);
        }

        // ---- epilogue: O / l -> bf16, staged in this tile's Q buffer (free:
        // o_final covers every MMA of the CTA that read it) in the
        // 128-byte-swizzled layout of the O tensor map, then two TMA stores.
        // LSE is a plain coalesced store.
        const size_t out_row = (static_cast<size_t>(b) * p.H + h) * p.N_q + row;
        if (has[t]) {
            ok = barrier_and(1 + t, 128, ok && mbar_wait(&c.o_final[t], 0, ctl));
            if (ok) {
                tc_fence_after_sync();
                const float inv_l = l > 0.f ? 1.0f / l : 0.f;
                uint8_t *stage = sQ + t * C::kQTileBytes;
                const int r = quad * 32 + lane;
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld_x32(tO + ch * 32, o);
                    uint8_t *dst_row = stage + (ch / 2) * kQChunkBytes + r * 128;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[8 * k]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
                        v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
                        v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
                        v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
                        const int c16 = (ch % 2) * 4 + k;          // 16-byte chunk within the 128-byte row
                        *reinterpret_cast<uint4 *>(dst_row + ((c16 ^ (r & 7)) << 4)) = v;
                    }
                }
                if (row_valid)
                    p.LSE[out_row] = l > 0.f ? (m_ref * cexp + __log2f(l)) * kLn2 : -INFINITY;
                fence_proxy_async_smem();
                named_barrier(1 + t, 128);
                if (quad == 0 && lane == 0) {
                    for (int ch = 0; ch < C::kChunks; ++ch)
                        tma_store_3d(&tmO, stage + ch * kQChunkBytes, ch * 64, r0[t], bh);
                    bulk_commit_group();
                    bulk_wait_all();        // stores complete before the CTA retires
                }
            }
        } else if (row_valid) {
            // No key is visible to any row of this tile.
            uint4 *dst = reinterpret_cast<uint4 *>(p.O + out_row * D);
            for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
            p.LSE[out_row] = -INFINITY;
        }
    }

    // ---- teardown (lanes 1-31 of warps 0 and 1 wait here for their lane 0)
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, C::kTmemCols);
    }
    if (threadIdx.x == 0) ATTN_TRACE_CLOCK(1);
}

template <int D, bool kSparse, int kT, int BN = kBN, bool kPf = (kT == 1)>
int launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to,
           const Params &p, int grid, const LaunchEnv &env, std::string &err)
{
    static std::atomic<uint64_t> configured{0};   // one bit per device
    const size_t smem = smem_bytes<D, kT, BN>();
    {
        cudaError_t e = set_smem_limit_once(reinterpret_cast<const void *>(attn_fwd_kernel<D, kSparse, kT, BN, kPf>),
                                            smem, configured);
        if (e != cudaSuccess) {
            err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
            return 5;
        }
    }
    attn_fwd_kernel<D, kSparse, kT, BN, kPf><<<grid, Cfg<D, kT, BN>::kThreads, smem, env.stream>>>(tq, tk, tv, to, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        err = std::string("attn_fwd launch: ") + cudaGetErrorString(e);
        return 5;
    }
    return 0;
}

// Writes O = 0, LSE = -inf for every row (used when N_kv == 0).
__global__ void fill_empty_kernel(__nv_bfloat16 *O, float *LSE, size_t rows, int d)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < rows;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        for (int k = 0; k < d; ++k) O[i * d + k] = __float2bfloat16(0.f);
        LSE[i] = -INFINITY;
    }
}

// Mean number of 128-key tiles a 128-row query tile visits (the host's copy
// of kv_range), which decides the form: long rows keep the tensor core busy
// best with two Q tiles ping-ponging in one CTA; short ones (windows, short
// causal problems) lose less to CTA start-up and drain with two one-tile
// CTAs per SM.
double mean_kv_tiles(int N_q, int N_kv, int lo_pad, int hi_pad)
{
    const long long off = static_cast<long long>(N_kv) - N_q;
    const int n = (N_q + kBM - 1) / kBM;
    long long total = 0;
    for (int qt = 0; qt < n; ++qt) {
        const long long r0 = static_cast<long long>(qt) * kBM, r1 = std::min<long long>(r0 + kBM, N_q);
        const long long key_lo = std::max(0LL, r0 + off - lo_pad);
        const long long key_hi = std::min(static_cast<long long>(N_kv), r1 - 1 + off + hi_pad + 1);
        if (key_hi > key_lo) total += (key_hi + kBN - 1) / kBN - key_lo / kBN;
    }
    return n > 0 ? static_cast<double>(total) / n : 0.0;
}

constexpr double kTwoTileMinKvTiles = 16.0;

}  // namespace

int launch_attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                    int H_kv, int N_q, int N_kv, int d, int causal, int window, float scale,
                    const uint8_t *block_mask, const LaunchEnv &env, std::string &err)
{
    if (N_q == 0 || B == 0) return 0;
    if (N_kv == 0) {
        const size_t rows = static_cast<size_t>(B) * H * N_q;
        fill_empty_kernel<<<static_cast<int>(std::min<size_t>((rows + 255) / 256, 4096)), 256, 0,
                            env.stream>>>(static_cast<__nv_bfloat16 *>(O), LSE, rows, d);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            err = std::string("fill launch: ") + cudaGetErrorString(e);
            return 5;
        }
        return 0;
    }
    Params p;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.B = B;
    p.H = H;
    p.H_kv = H_kv;
    p.N_q = N_q;
    p.N_kv = N_kv;
    constexpr int kNoPad = 1 << 30;
    if (causal) {
        p.hi_pad = 0;
        p.lo_pad = window > 0 ? window - 1 : kNoPad;
    } else {
        p.hi_pad = window > 0 ? window : kNoPad;   // symmetric local window
        p.lo_pad = window > 0 ? window : kNoPad;
    }
    p.group = H / H_kv;
    p.block_mask = block_mask;
    p.mask_qb = (N_q + kBM - 1) / kBM;
    p.mask_kb = (N_kv + kBN - 1) / kBN;
    // Q tiles per CTA (see Cfg).  Block-sparse launches use one: their density
    // is not known here, and sparse rows are short.
    const int kt = (!block_mask && mean_kv_tiles(N_q, N_kv, p.lo_pad, p.hi_pad) >= kTwoTileMinKvTiles) ? 2 : 1;
    // The dense one-tile form runs pipelined, on 64-key tiles (see Cfg).
    const int bn = (!block_mask && kt == 1) ? 64 : kBN;
    p.n_qblk = (N_q + kt * kBM - 1) / (kt * kBM);
    CUtensorMap tq, tk, tv, to;
    if (!make_tma_bf16_3d(tq, Q, d, N_q, static_cast<uint64_t>(B) * H, kBM, err) ||
        !make_tma_bf16_3d(to, O, d, N_q, static_cast<uint64_t>(B) * H, kBM, err) ||
        !make_tma_bf16_3d(tk, K, d, N_kv, static_cast<uint64_t>(B) * H_kv, bn, err) ||
        !make_tma_bf16_3d(tv, V, d, N_kv, static_cast<uint64_t>(B) * H_kv, bn, err))
        return 5;
    p.c = scale * 1.4426950408889634f;
    p.inject = env.inject;
    // Q prefetch for the next block on an SM: in the one-tile forms (two CTAs
    // per SM) and in the two-tile form for grouped heads, whose K / V mostly
    // hit L2 already.  Measured kernel-only: causal window 256 +2.4 %, causal
    // 2k +1-2 %, block-sparse +0.4 %, GQA 8k causal +1.4 %, symmetric window 256
    // unchanged; in the two-tile form for MHA the 16k causal shape lost 0.2 %
    // with it (its K / V prefixes already overflow L2).  (Not at d = 64, whose
    // two-tile producer spills registers with the prefetch code.)
    const bool pf2 = p.group > 1 && d == 128;
    p.pf_stride = kt == 1 ? 2 * env.num_sms : (pf2 ? env.num_sms : 0);
    p.status = env.status;
    p.timeout_ns = env.timeout_ns;
    const long long grid = static_cast<long long>(p.n_qblk) * B * H;
    if (grid > 0x7fffffffLL) {
        err = "attn_fwd: problem too large for one launch";
        return 2;
    }
    const int g = static_cast<int>(grid);
    // Block-sparse launches keep the one-tile form on 128-key tiles: the
    // pipelined 64-key form (which also walks a block mask) measured 11 % slower
    // at 25 % density, its scattered tiles paying the N = 64 score MMAs.
    if (block_mask)
        return d == 128 ? launch<128, true, 1>(tq, tk, tv, to, p, g, env, err)
                        : launch<64, true, 1>(tq, tk, tv, to, p, g, env, err);
    if (kt == 1)
        return d == 128 ? launch<128, false, 1, 64>(tq, tk, tv, to, p, g, env, err)
                        : launch<64, false, 1, 64>(tq, tk, tv, to, p, g, env, err);
    if (pf2) return launch<128, false, 2, kBN, true>(tq, tk, tv, to, p, g, env, err);
    return d == 128 ? launch<128, false, 2>(tq, tk, tv, to, p, g, env, err)
                    : launch<64, false, 2>(tq, tk, tv, to, p, g, env, err);
}

int attn_trace_fetch(void *host, size_t bytes, std::string &err)
{
#ifdef GBATTN_TRACE
    static_assert(kAtEvents == GBATTN_ATTN_TRACE_EVENTS && kAtTiles == GBATTN_ATTN_TRACE_TILES &&
                      kAtCtas == GBATTN_ATTN_TRACE_CTAS,
                  "trace layout of the public header");
    constexpr size_t n0 = sizeof(g_attn_trace), n1 = sizeof(g_attn_trace_clock);
    static_assert(n0 + n1 == GBATTN_ATTN_TRACE_BYTES, "trace size of the public header");
    if (host == nullptr || bytes < n0 + n1) {
        err = "gbattn_attn_trace: host buffer missing or smaller than GBATTN_ATTN_TRACE_BYTES";
        return GBATTN_ERR_INVALID_ARG;
    }
    void *d0 = nullptr, *d1 = nullptr;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(host, g_attn_trace, n0);
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(static_cast<char *>(host) + n0, g_attn_trace_clock, n1);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&d0, g_attn_trace);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&d1, g_attn_trace_clock);
    if (e == cudaSuccess) e = cudaMemset(d0, 0, n0);
    if (e == cudaSuccess) e = cudaMemset(d1, 0, n1);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        err = std::string("gbattn_attn_trace: ") + cudaGetErrorString(e);
        return GBATTN_ERR_LAUNCH;
    }
    return GBATTN_OK;
#else
    (void)host;
    (void)bytes;
    err = "gbattn_attn_trace: this library was built without GBATTN_TRACE";
    return GBATTN_ERR_UNSUPPORTED;
#endif
}

}  // namespace gbattn
