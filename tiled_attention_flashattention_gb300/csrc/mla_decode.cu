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
//   CTA 0 holds latent dims [0, 256): its Q part and KV tiles cover those
//         dims; it computes the partial score over them and owns O[:, 0:256);
//   CTA 1 holds latent dims [256, 512) plus the 64 RoPE dims, computes the
//         partial score over those 320 dims and owns O[:, 256:512).
// Every KV byte is read from HBM by exactly one CTA.  The two fp32 partial
// score tiles (128 heads x 64 keys, 32 KB) are swapped with one bulk copy per
// CTA per tile (TMA engine, shared memory to the peer's shared memory), so
// both CTAs hold the same full score tile and run the same online softmax;
// each then multiplies P by its own latent half (V = KV_latent).
//
// Work split: the B * ceil(N_kv / 64) key tiles are cut into one contiguous
// range per cluster (as many clusters as fit on the GPU at once).  A range
// that covers a whole sequence writes the final O and LSE; a partial range
// writes O / l and its LSE to the workspace, and a small combine kernel merges
// the pieces of each split sequence with the exact log-sum-exp rule
// (TileLang 学习笔记, "Online Softmax 的关键", applied across key ranges).
// Only the first and the last sequence of a cluster's range can be partial,
// so the workspace holds two slots per cluster whatever B and N_kv are.
//
// Per CTA (384 threads, one CTA per SM):
//   warp 0      TMA producer: this CTA's dims of each 64-key tile, 4 stages;
//   warp 1      tcgen05 issuer: S_part = Q_part K_part^T with Q from TMEM,
//               then O_half += P V_half with P from TMEM (N = 256);
//   warps 4-7   exchange (one thread per head): this sequence's Q part into
//               TMEM; per tile read S_part, send it to the peer, add the
//               peer's part, hand the full score row to the softmax warps;
//   warps 8-11  softmax (one thread per head): online softmax, P (bf16) into
//               TMEM, O rescaling, epilogue.
// The exchange of tile j+1 overlaps the softmax of tile j; the score buffer
// is released as soon as the exchange warps have read it.
// TMEM: O half [0, 256), S [256, 320), P [320, 352), Q part [352, 512).
#include <cmath>
#include <cstdio>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kH = 128;                   // heads per tile (MMA M)
constexpr int kBN = 64;                   // keys per tile
constexpr int kDc = 512;
constexpr int kHalf = 256;                // latent dims owned by one CTA
constexpr int kKvChunk = kBN * 128;       // [64 keys x 64 dims] bf16, one TMA box
constexpr int kMaxChunks = 5;             // contraction chunks of CTA 1 (4 latent + RoPE)
constexpr int kStageBytes = kMaxChunks * kKvChunk;
constexpr int kStages = 4;
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;
constexpr uint32_t kColP = 320;
constexpr uint32_t kColQ = 352;
constexpr int kXBytes = kH * kBN * 4;     // one partial score tile (fp32)
constexpr uint32_t kBarX = 1, kBarS = 2;  // named barriers of the exchange / softmax warps
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;

struct Ctl {
    uint64_t q_full, q_empty;
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full, s_free;
    uint64_t xfull, xfree, sready;
    uint64_t p_full, pfree;
    uint64_t o_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes =
    1024 + static_cast<size_t>(kStages) * kStageBytes + 2 * static_cast<size_t>(kXBytes) + sizeof(Ctl);

struct Params {
    const __nv_bfloat16 *Qn;   // [B][128][512]
    const __nv_bfloat16 *Qp;   // [B][128][64]
    __nv_bfloat16 *O;
    float *LSE;
    float *ws_O;        // [slots][128][512] fp32, O / l of partial ranges
    float *ws_LSE;      // [slots][128]
    int B, N_kv, ntile;
    long long T;        // B * ntile
    int C;              // clusters
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

// The cluster whose range holds flat tile x.
__host__ __device__ __forceinline__ int cluster_of_tile(long long x, long long T, int C)
{
    return static_cast<int>(((x + 1) * C - 1) / T);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_split_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ CUtensorMap tmKp,
                     const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sKV = smem;                                   // [stage][chunk][64 keys][128 B]
    uint8_t *sSend = sKV + kStages * kStageBytes;          // [128 rows][256 B] fp32, swizzled
    uint8_t *sRecv = sSend + kXBytes;                      // [128 rows][256 B] fp32, swizzled
    Ctl &c = *reinterpret_cast<Ctl *>(sRecv + kXBytes);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
    const int cl = blockIdx.x / 2;
    const long long t_begin = range_start(cl, p.T, p.C), t_end = range_start(cl + 1, p.T, p.C);
    const int nch = rank == 0 ? 4 : 5;              // contraction chunks of this CTA
    const int dim0 = static_cast<int>(rank) * kHalf;
    const int b_first = static_cast<int>(t_begin / p.ntile);
    const int b_last = t_end > t_begin ? static_cast<int>((t_end - 1) / p.ntile) : b_first - 1;

    if (threadIdx.x == 0) {
        mbar_init(&c.q_full, 128);
        mbar_init(&c.q_empty, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&c.full[s], 1);
            mbar_init(&c.empty[s], 1);
        }
        mbar_init(&c.s_full, 1);
        mbar_init(&c.s_free, 128);
        mbar_init(&c.xfull, 1);       // this CTA's expect_tx arrive + the peer's 32 KB
        mbar_init(&c.xfree, 1);       // remote arrive: the peer's receive buffer is free
        mbar_init(&c.sready, 128);
        mbar_init(&c.p_full, 128);
        mbar_init(&c.pfree, 1);
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

    if (warp == 0) {
        // =================== TMA producer ===================
        if (lane == 0) {
            tma_prefetch_desc(&tmKV);
            tma_prefetch_desc(&tmKp);
            bool ok = true;
            int it = 0;
            const uint32_t kvbytes = nch * kKvChunk;
            for (int b = b_first; b <= b_last && ok; ++b) {
                const long long x0 = max(t_begin, static_cast<long long>(b) * p.ntile);
                const long long x1 = min(t_end, static_cast<long long>(b + 1) * p.ntile);
                for (long long x = x0; x < x1; ++x) {
                    const int key0 = static_cast<int>(x - static_cast<long long>(b) * p.ntile) * kBN;
                    const int s = it % kStages;
                    const uint32_t round = static_cast<uint32_t>(it / kStages);
                    if (round > 0 && !(ok = mbar_wait(&c.empty[s], (round & 1u) ^ 1u, ctl))) break;
                    uint8_t *dst = sKV + s * kStageBytes;
                    mbar_arrive_expect_tx(&c.full[s], kvbytes);
                    for (int ch = 0; ch < 4; ++ch)
                        tma_load_3d(dst + ch * kKvChunk, &tmKV, &c.full[s], dim0 + ch * 64, key0, b);
                    if (rank == 1) tma_load_3d(dst + 4 * kKvChunk, &tmKp, &c.full[s], 0, key0, b);
                    ++it;
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                const WaitCtl drain{&no_abort, p.status, p.timeout_ns};
                for (int i = (it > kStages ? it - kStages : 0); i < it; ++i)
                    mbar_wait(&c.full[i % kStages], static_cast<uint32_t>(i / kStages) & 1u, drain);
            }
        }
    } else if (warp == 1) {
        // =================== tensor-core issuer ===================
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kH, kBN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(kH, kHalf, false, true);
            const uint32_t sKVa = smem_u32(sKV);
            bool ok = true;
            int it = 0, seg = 0;
            uint32_t g = 0;      // global tile counter
            // O_half += P V_half for tile gp: P from TMEM (8 columns per 16
            // keys); V = the latent chunks of stage sp read N-major (64-dim
            // blocks 8 KB apart, 16 keys = 2 KB per MMA).
            auto issue_pv = [&](uint32_t gp, int sp, bool first) -> bool {
                if (!mbar_wait(&c.p_full, gp & 1u, ctl)) return false;
                if (first && seg > 0 && !mbar_wait(&c.o_empty, (seg - 1) & 1, ctl)) return false;
                tc_fence_after_sync();
                const uint64_t vd = smem_desc_sw128(sKVa + sp * kStageBytes, kKvChunk, 1024);
                umma_ts(tbase + kColO, tbase + kColP, vd, idPV, first ? 0u : 1u);
#pragma unroll
                for (int k = 1; k < kBN / 16; ++k)
                    umma_ts(tbase + kColO, tbase + kColP + k * 8, desc_advance(vd, k * 2048), idPV, 1u);
                umma_commit(&c.pfree);
                umma_commit(&c.empty[sp]);
                return true;
            };
            for (int b = b_first; b <= b_last && ok; ++b, ++seg) {
                const long long x0 = max(t_begin, static_cast<long long>(b) * p.ntile);
                const long long x1 = min(t_end, static_cast<long long>(b + 1) * p.ntile);
                const int n = static_cast<int>(x1 - x0);
                if (!(ok = mbar_wait(&c.q_full, seg & 1, ctl))) break;
                int prev_stage = -1;
                for (int i = 0; i < n; ++i) {
                    const int s = it % kStages;
                    if (!(ok = mbar_wait(&c.full[s], static_cast<uint32_t>(it / kStages) & 1u, ctl))) break;
                    if (g > 0 && !(ok = mbar_wait(&c.s_free, (g - 1) & 1u, ctl))) break;
                    tc_fence_after_sync();
                    // S_part = Q_part K_part^T: Q from TMEM (8 columns per 16 dims).
                    const uint64_t kvd = smem_desc_sw128(sKVa + s * kStageBytes, 16, 1024);
                    umma_ts(tbase + kColS, tbase + kColQ, kvd, idS, 0u);
                    for (int k = 1; k < nch * 4; ++k)
                        umma_ts(tbase + kColS, tbase + kColQ + k * 8,
                                desc_advance(kvd, (k / 4) * kKvChunk + (k % 4) * 32), idS, 1u);
                    umma_commit(&c.s_full);
                    if (i == n - 1) umma_commit(&c.q_empty);
                    if (i > 0 && !(ok = issue_pv(g - 1, prev_stage, i == 1))) break;
                    prev_stage = s;
                    ++it;
                    ++g;
                }
                if (ok && n > 0) ok = issue_pv(g - 1, prev_stage, n == 1);
            }
            umma_commit(&c.drain);
            volatile int no_abort = 0;
            const WaitCtl drain{&no_abort, p.status, p.timeout_ns};
            mbar_wait(&c.drain, 0, drain);
        }
    } else if (warp >= 4 && warp < 8) {
        // =================== Q load + partial-score exchange (one thread per head) ===================
        const int quad = warp - 4;
        const int row = quad * 32 + lane;
        const bool leader = threadIdx.x == 128;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t swz = static_cast<uint32_t>(row & 15);
        const uint32_t peer_recv = mapa_shared(smem_u32(sRecv), peer);
        const uint32_t peer_xfull = mapa_shared(smem_u32(&c.xfull), peer);
        float4 *send_row = reinterpret_cast<float4 *>(sSend + row * 256);
        float4 *recv_row = reinterpret_cast<float4 *>(sRecv + row * 256);
        bool ok = true;
        uint32_t g = 0;
        int seg = 0;
        for (int b = b_first; b <= b_last && ok; ++b, ++seg) {
            const long long x0 = max(t_begin, static_cast<long long>(b) * p.ntile);
            const long long x1 = min(t_end, static_cast<long long>(b + 1) * p.ntile);
            const int n = static_cast<int>(x1 - x0);
            // This CTA's part of the query row into TMEM (two bf16 per column).
            if (seg > 0 && !(ok = barrier_and(kBarX, 128, mbar_wait(&c.q_empty, (seg - 1) & 1, ctl)))) break;
            const uint4 *qn = reinterpret_cast<const uint4 *>(p.Qn + (static_cast<size_t>(b) * kH + row) * kDc + dim0);
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t r[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 v = __ldg(qn + ch * 8 + k);
                    r[4 * k] = v.x;
                    r[4 * k + 1] = v.y;
                    r[4 * k + 2] = v.z;
                    r[4 * k + 3] = v.w;
                }
                tmem_st_x32(tbase + lane_base + kColQ + ch * 32, r);
            }
            if (rank == 1) {
                const uint4 *qp = reinterpret_cast<const uint4 *>(p.Qp + (static_cast<size_t>(b) * kH + row) * 64);
                uint32_t r[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 v = __ldg(qp + k);
                    r[4 * k] = v.x;
                    r[4 * k + 1] = v.y;
                    r[4 * k + 2] = v.z;
                    r[4 * k + 3] = v.w;
                }
                tmem_st_x32(tbase + lane_base + kColQ + 128, r);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&c.q_full);

            for (int i = 0; i < n; ++i, ++g) {
                if (!(ok = barrier_and(kBarX, 128, mbar_wait(&c.s_full, g & 1u, ctl)))) break;
                tc_fence_after_sync();
                uint32_t sr[64];
                tmem_ld_x64(tbase + lane_base + kColS, sr);
                tc_fence_before_sync();
                mbar_arrive(&c.s_free);
                // The previous copy must have finished reading the send buffer.
                if (leader && g > 0) bulk_wait_read_all();
                named_barrier(kBarX, 128);
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    send_row[q ^ swz] = make_float4(__uint_as_float(sr[4 * q]), __uint_as_float(sr[4 * q + 1]),
                                                    __uint_as_float(sr[4 * q + 2]), __uint_as_float(sr[4 * q + 3]));
                fence_proxy_async_smem();      // the copy engine reads the send buffer
                named_barrier(kBarX, 128);
                if (leader) {
                    // The peer's receive buffer is free once its softmax warps read tile g - 1.
                    bool got = (g == 0) || mbar_wait_cluster(&c.xfree, (g - 1) & 1u, ctl);
                    if (got) {
                        mbar_arrive_expect_tx(&c.xfull, kXBytes);   // this CTA's incoming tile
                        bulk_copy_to_peer(peer_recv, sSend, kXBytes, peer_xfull);
                        bulk_commit_group();
                    }
                }
                if (!(ok = barrier_and(kBarX, 128, mbar_wait_cluster(&c.xfull, g & 1u, ctl)))) break;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    float4 v = recv_row[q ^ swz];
                    v.x += __uint_as_float(sr[4 * q]);
                    v.y += __uint_as_float(sr[4 * q + 1]);
                    v.z += __uint_as_float(sr[4 * q + 2]);
                    v.w += __uint_as_float(sr[4 * q + 3]);
                    recv_row[q ^ swz] = v;
                }
                mbar_arrive(&c.sready);
            }
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
        const uint32_t swz = static_cast<uint32_t>(row & 15);
        const uint32_t peer_xfree = mapa_shared(smem_u32(&c.xfree), peer);
        const float4 *recv_row = reinterpret_cast<const float4 *>(sRecv + row * 256);
        bool ok = true;
        uint32_t g = 0;
        int seg = 0;
        for (int b = b_first; b <= b_last && ok; ++b, ++seg) {
            const long long x0 = max(t_begin, static_cast<long long>(b) * p.ntile);
            const long long x1 = min(t_end, static_cast<long long>(b + 1) * p.ntile);
            const int n = static_cast<int>(x1 - x0);
            float m_ref = -INFINITY, l = 0.f;
            for (int i = 0; i < n; ++i, ++g) {
                const bool got = mbar_wait(&c.sready, g & 1u, ctl);
                float s[64];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float4 v = recv_row[q ^ swz];
                    s[4 * q] = v.x;
                    s[4 * q + 1] = v.y;
                    s[4 * q + 2] = v.z;
                    s[4 * q + 3] = v.w;
                }
                // all 128 rows read: the peer may send its next tile
                if (!(ok = barrier_and(kBarS, 128, got))) break;
                if (leader) mbar_arrive_remote(peer_xfree);

                const int key0 = static_cast<int>(x0 + i - static_cast<long long>(b) * p.ntile) * kBN;
                if (key0 + kBN > p.N_kv) {
#pragma unroll
                    for (int k = 0; k < 64; ++k)
                        if (key0 + k >= p.N_kv) s[k] = -INFINITY;
                }
                float mx = s[0];
#pragma unroll
                for (int k = 1; k < 64; ++k) mx = fmaxf(mx, s[k]);
                const bool move = mx > m_ref + thr;
                const float new_ref = move ? mx : m_ref;
                const float alpha = move ? ex2_approx((m_ref - new_ref) * cexp) : 1.0f;
                m_ref = new_ref;
                const float base = (m_ref == -INFINITY) ? 0.f : m_ref * cexp;
                float sum = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float p0 = ex2_approx(fmaf(s[2 * k], cexp, -base));
                    const float p1 = ex2_approx(fmaf(s[2 * k + 1], cexp, -base));
                    sum += p0 + p1;
                    pk[k] = pack_bf16x2(p0, p1);
                }
                l = l * alpha + sum;
                // PV of the previous tile must be done: it read the P buffer,
                // and O must be stable before it is rescaled.
                if (g > 0 && !(ok = barrier_and(kBarS, 128, mbar_wait(&c.pfree, (g - 1) & 1u, ctl)))) break;
                tc_fence_after_sync();
                if (i > 0 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
                    for (int ch = 0; ch < kHalf / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld_x32(tO + ch * 32, o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st_x32(tO + ch * 32, o);
                    }
                }
                tmem_st_x32(tbase + lane_base + kColP, pk);
                tmem_st_wait();
                tc_fence_before_sync();
                mbar_arrive(&c.p_full);
            }
            if (!ok) break;

            // ---- epilogue of this range of sequence b (after its last PV)
            if (!(ok = barrier_and(kBarS, 128, mbar_wait(&c.pfree, (g - 1) & 1u, ctl)))) break;
            tc_fence_after_sync();
            const bool whole = (n == p.ntile);
            const float inv_l = l > 0.f ? 1.0f / l : 0.f;
            const float lse = l > 0.f ? (m_ref * cexp + __log2f(l)) * kLn2 : -INFINITY;
            const size_t slot = static_cast<size_t>(cl) * 2 + (b == b_first ? 0 : 1);
#pragma unroll 1
            for (int ch = 0; ch < kHalf / 32; ++ch) {
                uint32_t o[32];
                tmem_ld_x32(tO + ch * 32, o);
                if (whole) {
                    uint4 v[4];
                    uint32_t *w = reinterpret_cast<uint32_t *>(v);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        w[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
                    uint4 *dst = reinterpret_cast<uint4 *>(p.O + (static_cast<size_t>(b) * kH + row) * kDc +
                                                           dim0 + ch * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) dst[k] = v[k];
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(p.ws_O + (slot * kH + row) * kDc + dim0 + ch * 32);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv_l, __uint_as_float(o[4 * k + 1]) * inv_l,
                                             __uint_as_float(o[4 * k + 2]) * inv_l,
                                             __uint_as_float(o[4 * k + 3]) * inv_l);
                }
            }
            if (rank == 0) {
                if (whole)
                    p.LSE[static_cast<size_t>(b) * kH + row] = lse;
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

// Merge the partial ranges of each split sequence: LSE = ln sum_s e^{LSE_s},
// O = sum_s e^{LSE_s - LSE} O_s.  One block per (sequence, group of 16
// heads), 256 threads, 32 output dims per thread; sequences written whole by
// the split kernel are skipped.
__global__ void __launch_bounds__(256) mla_combine_kernel(const Params p)
{
    const int b = blockIdx.x / 8, hg = blockIdx.x % 8;
    const long long x0 = static_cast<long long>(b) * p.ntile;
    const int c0 = cluster_of_tile(x0, p.T, p.C);
    const int c1 = cluster_of_tile(x0 + p.ntile - 1, p.T, p.C);
    if (c0 == c1) return;
    const int h = hg * 16 + threadIdx.x / 16;
    const int d0 = (threadIdx.x % 16) * 32;
    float mx = -INFINITY;
    for (int q = c0; q <= c1; ++q) {
        const size_t slot = static_cast<size_t>(q) * 2 + (b == range_start(q, p.T, p.C) / p.ntile ? 0 : 1);
        mx = fmaxf(mx, p.ws_LSE[slot * kH + h]);
    }
    float denom = 0.f;
    for (int q = c0; q <= c1; ++q) {
        const size_t slot = static_cast<size_t>(q) * 2 + (b == range_start(q, p.T, p.C) / p.ntile ? 0 : 1);
        denom += expf(p.ws_LSE[slot * kH + h] - mx);
    }
    const float lse = mx + logf(denom);
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
    for (int q = c0; q <= c1; ++q) {
        const size_t slot = static_cast<size_t>(q) * 2 + (b == range_start(q, p.T, p.C) / p.ntile ? 0 : 1);
        const float w = expf(p.ws_LSE[slot * kH + h] - lse);
        const float4 *src = reinterpret_cast<const float4 *>(p.ws_O + (slot * kH + h) * kDc + d0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = src[k];
            acc[4 * k] += w * v.x;
            acc[4 * k + 1] += w * v.y;
            acc[4 * k + 2] += w * v.z;
            acc[4 * k + 3] += w * v.w;
        }
    }
    uint4 out[4];
    uint32_t *o = reinterpret_cast<uint32_t *>(out);
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = pack_bf16x2(acc[2 * k], acc[2 * k + 1]);
    uint4 *dst = reinterpret_cast<uint4 *>(p.O + (static_cast<size_t>(b) * kH + h) * kDc + d0);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = out[k];
    if (threadIdx.x % 16 == 0) p.LSE[static_cast<size_t>(b) * kH + h] = lse;
}

struct Plan {
    int ntile, C, max_seg;
    long long T;
    size_t slots;
};

// Cluster count: as many 2-CTA clusters as are co-resident on the device
// (queried once per process), never more than the number of key tiles.
int resident_clusters(int num_sms)
{
    static int cached = -1;
    if (cached > 0) return cached;
    int n = 0;
    if (cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
        if (cudaOccupancyMaxActiveClusters(&n, mla_split_kernel, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    if (n <= 0) n = num_sms / 2;
    cached = n;
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
    return pl.slots * kH * kDc * sizeof(float) + pl.slots * kH * sizeof(float);
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
// SMs: 80 two-CTA clusters x 2 partial slots x (128 x 512 fp32 O + 128 fp32
// LSE) = 42,024,960 bytes.  Every GPU that loads the library holds it until
// the process exits.
constexpr size_t kNoAllocMaxClusters = 80;
constexpr size_t kNoAllocScratchBytes =
    kNoAllocMaxClusters * 2 * (static_cast<size_t>(kH) * kDc * sizeof(float) + kH * sizeof(float));
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

size_t mla_workspace_bytes(int B, int H, int N_kv, int d_c, int num_sms)
{
    if (B < 1 || H != kH || N_kv < 1 || d_c != kDc) return 0;
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
    CUtensorMap tkv, tkp;
    if (!make_tma_bf16_3d(tkv, KV_latent, d_c, N_kv, B, kBN, err) || !make_tma_bf16_3d(tkp, K_pe, d_r, N_kv, B, kBN, err))
        return 5;
    Params p;
    p.Qn = static_cast<const __nv_bfloat16 *>(Q_nope);
    p.Qp = static_cast<const __nv_bfloat16 *>(Q_pe);
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.LSE = LSE;
    p.ws_O = static_cast<float *>(workspace);
    p.ws_LSE = p.ws_O + pl.slots * kH * kDc;
    p.B = B;
    p.N_kv = N_kv;
    p.ntile = pl.ntile;
    p.T = pl.T;
    p.C = pl.C;
    p.max_seg = pl.max_seg;
    p.c = scale * 1.4426950408889634f;
    p.status = env.status;
    p.timeout_ns = env.timeout_ns;
    cudaError_t e = cudaFuncSetAttribute(mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e == cudaSuccess) {
        mla_split_kernel<<<2 * pl.C, kThreads, kSmemBytes, env.stream>>>(tkv, tkp, p);
        e = cudaGetLastError();
    }
    bool split = false;   // does a cluster range boundary fall inside a sequence?
    for (int cl = 1; cl < pl.C && !split; ++cl) split = range_start(cl, pl.T, pl.C) % pl.ntile != 0;
    if (e == cudaSuccess && split) {
        mla_combine_kernel<<<B * 8, 256, 0, env.stream>>>(p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        err = std::string("mla_decode launch: ") + cudaGetErrorString(e);
        return 5;
    }
    return 0;
}

}  // namespace gbattn
