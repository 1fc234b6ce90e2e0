// selftest.cu -- one-tile check of the tensor-core operand layouts used by the
// attention kernels:
//   S = A B^T : A, B K-major, TMA-loaded with 128-byte swizzle (as Q and K);
//   O = P V   : P written to TMEM as bf16 pairs from registers (as the softmax
//               writes P over S), V TMA-loaded and read N-major (as V tiles).
// 128 threads; TMEM: S in columns [0,128) (P later overwrites [0,64)), O in
// [128,256).
#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kTile = 128 * 128 * 2;       // one 128x128 bf16 tile
constexpr int kChunk = 128 * 128;          // 128 rows x 128 B

struct StCtl {
    uint64_t tma;
    uint64_t mma;
    uint32_t tmem_base;
    int abort;
};

__global__ void __launch_bounds__(128, 1)
    selftest_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmV, const uint32_t *P, float *S, float *O,
                    int *status, uint64_t timeout_ns)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem, *sB = smem + kTile, *sV = smem + 2 * kTile;
    StCtl &c = *reinterpret_cast<StCtl *>(smem + 3 * kTile);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        mbar_init(&c.tma, 1);
        mbar_init(&c.mma, 1);
        c.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&c.tmem_base, 256);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tbase = c.tmem_base;
    const WaitCtl ctl{&c.abort, status, timeout_ns};
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int row = warp * 32 + lane;

    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&c.tma, 3 * kTile);
        for (int ch = 0; ch < 2; ++ch) {
            tma_load_3d(sA + ch * kChunk, &tmA, &c.tma, ch * 64, 0, 0);
            tma_load_3d(sB + ch * kChunk, &tmB, &c.tma, ch * 64, 0, 0);
            tma_load_3d(sV + ch * kChunk, &tmV, &c.tma, ch * 64, 0, 0);
        }
        if (mbar_wait(&c.tma, 0, ctl)) {
            const uint32_t id = idesc_bf16_f32(128, 128, false, false);
            for (int k = 0; k < 8; ++k) {
                const uint32_t koff = (k / 4) * kChunk + (k % 4) * 32;
                umma_ss(tbase, smem_desc_sw128(smem_u32(sA) + koff, 16, 1024),
                        smem_desc_sw128(smem_u32(sB) + koff, 16, 1024), id, k > 0);
            }
        }
        umma_commit(&c.mma);
    }
    __syncwarp();
    bool ok = __all_sync(0xffffffffu, mbar_wait(&c.mma, 0, ctl));
    if (ok) {
        tc_fence_after_sync();
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t r[32];
            tmem_ld_x32(tbase + lane_base + ch * 32, r);
            for (int i = 0; i < 32; ++i) S[row * 128 + ch * 32 + i] = __uint_as_float(r[i]);
        }
        // P row -> TMEM columns [0, 64) as bf16 pairs
        for (int ch = 0; ch < 2; ++ch) {
            uint32_t r[32];
            for (int i = 0; i < 32; ++i) r[i] = P[row * 64 + ch * 32 + i];
            tmem_st_x32(tbase + lane_base + ch * 32, r);
        }
        tmem_st_wait();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {
        tc_fence_after_sync();
        if (ok && !c.abort) {
            const uint32_t id = idesc_bf16_f32(128, 128, false, true);
            for (int k = 0; k < 8; ++k)
                umma_ts(tbase + 128, tbase + k * 8,
                        smem_desc_sw128(smem_u32(sV) + k * 2048, kChunk, 1024), id, k > 0);
        }
        umma_commit(&c.mma);
    }
    __syncwarp();
    ok = __all_sync(0xffffffffu, mbar_wait(&c.mma, 1, ctl)) && ok;
    if (ok) {
        tc_fence_after_sync();
        for (int ch = 0; ch < 4; ++ch) {
            uint32_t r[32];
            tmem_ld_x32(tbase + lane_base + 128 + ch * 32, r);
            for (int i = 0; i < 32; ++i) O[row * 128 + ch * 32 + i] = __uint_as_float(r[i]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tbase, 256);
    }
}

}  // namespace

int launch_selftest_umma(const void *A, const void *B, const void *P, const void *V, float *S,
                         float *O, const LaunchEnv &env, std::string &err)
{
    CUtensorMap ta, tb, tv;
    if (!make_tma_bf16_3d(ta, A, 128, 128, 1, 128, err) ||
        !make_tma_bf16_3d(tb, B, 128, 128, 1, 128, err) ||
        !make_tma_bf16_3d(tv, V, 128, 128, 1, 128, err))
        return 5;
    const size_t smem = 1024 + 3 * kTile + sizeof(StCtl);
    cudaError_t e = cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e == cudaSuccess) {
        selftest_kernel<<<1, 128, smem, env.stream>>>(ta, tb, tv, static_cast<const uint32_t *>(P), S,
                                                      O, env.status, env.timeout_ns);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        err = std::string("selftest launch: ") + cudaGetErrorString(e);
        return 5;
    }
    return 0;
}

}  // namespace gbattn
