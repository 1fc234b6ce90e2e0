// probes.cu -- micro-benchmarks of the GB300 facts the kernels' design rests on
// (a measurement tool, not part of libgbattn.so): per-SM instruction rates of
// the softmax's instruction mix, the issue rate of back-to-back tcgen05.mma by
// shape, and single-thread synchronisation latencies.  Every wait is bounded;
// every access stays inside the buffers allocated here.  Built and run by
// `python -m tiled_attention_flashattention_gb300.probes`.
#include <cstdio>
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

using namespace gbattn;

namespace {

// ---------------------------------------------------------------------------
// Instruction rates: each thread runs 8 independent chains of one instruction.
template <int OP>
__global__ void __launch_bounds__(512, 1) alu_rate(float *out, long long *cyc, int iters, float seed)
{
    float v[8], w[8], v2[8];
    uint64_t pr[8], q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = seed * (i + 1) * 1e-3f - 0.5f;
        w[i] = seed * (i + 3) * 1e-3f;
        v2[i] = w[i] + 0.25f;
        pr[i] = f2_pack(v[i], w[i]);
        q[i] = f2_pack(w[i], v[i]);
    }
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if constexpr (OP == 0) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(v[i]));
            if constexpr (OP == 1) asm volatile("max.f32 %0, %0, %1;" : "+f"(v[i]) : "f"(w[i]));
            if constexpr (OP == 2) asm volatile("max.f32 %0, %0, %1, %2;" : "+f"(v[i]) : "f"(w[i]), "f"(w[(i + 3) & 7]));
            if constexpr (OP == 3) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(v[i]) : "f"(w[i]), "f"(w[(i + 1) & 7]));
            if constexpr (OP == 4) asm volatile("add.rn.f32 %0, %0, %1;" : "+f"(v[i]) : "f"(w[i]));
            if constexpr (OP == 5) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(pr[i]) : "l"(q[i]), "l"(q[(i + 1) & 7]));
            if constexpr (OP == 6) asm volatile("add.rn.f32x2 %0, %0, %1;" : "+l"(pr[i]) : "l"(q[i]));
            if constexpr (OP == 7) {
                asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(v[i]));
                asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(v2[i]) : "f"(w[i]), "f"(w[(i + 1) & 7]));
            }
        }
    }
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float a, b;
        f2_unpack(pr[i], a, b);
        s += v[i] + v2[i] + a + b;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    if (threadIdx.x % 32 == 0) cyc[blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32] = t1 - t0;
}

template <int OP>
void run_alu(const char *name, int sms, float *out, long long *cyc)
{
    const int iters = 4096, threads = 512;
    static long long h[152 * 16];
    for (int rep = 0; rep < 2; ++rep) alu_rate<OP><<<sms, threads>>>(out, cyc, iters, 1.0f);
    if (cudaDeviceSynchronize() != cudaSuccess) { printf("%s: %s\n", name, cudaGetErrorString(cudaGetLastError())); return; }
    const int nw = threads / 32;
    cudaMemcpy(h, cyc, sizeof(long long) * sms * nw, cudaMemcpyDeviceToHost);
    long long mx = 1;
    for (int i = 0; i < sms * nw; ++i) mx = h[i] > mx ? h[i] : mx;
    printf("  %-36s %7.1f per cycle per SM\n", name, double(threads) * iters * 8 / mx);
}

// ---------------------------------------------------------------------------
// Shared memory of the tensor-core and latency probes: a 16 KB A tile (128 rows
// x 128 B), a 32 KB B tile (256 rows x 128 B, or two 16 KB N-major chunks),
// eight mbarriers, the TMEM base and an abort flag.
constexpr int kProbeSmem = 1024 + 49152 + 128;

struct ProbeSmem {
    uint8_t *a, *b;
    uint64_t *bar;
    uint32_t *tmem_base;
    volatile int *abort;
};

__device__ ProbeSmem probe_setup(uint8_t *raw)
{
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    ProbeSmem m{smem, smem + 16384, reinterpret_cast<uint64_t *>(smem + 49152),
                reinterpret_cast<uint32_t *>(smem + 49152 + 64), reinterpret_cast<volatile int *>(smem + 49152 + 72)};
    for (int i = threadIdx.x; i < 49152 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(smem)[i] = 0x3c003c00u;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(&m.bar[i], 1);
        *m.abort = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    if (threadIdx.x / 32 == 0) {
        tmem_alloc(m.tmem_base, 512);
        tmem_relinquish();
        tc_fence_before_sync();
    }
    __syncthreads();
    tc_fence_after_sync();
    return m;
}

__device__ void probe_teardown(uint32_t tb)
{
    __syncthreads();
    if (threadIdx.x / 32 == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tb, 512);
    }
}

// Back-to-back MMAs from one thread: cycles per MMA while issuing, and until the
// last one completes.
template <int MODE>
__global__ void __launch_bounds__(128, 1) mma_rate(long long *out, int nmma, int *status)
{
    extern __shared__ uint8_t raw[];
    const ProbeSmem m = probe_setup(raw);
    const uint32_t tb = *m.tmem_base;
    if (threadIdx.x == 0) {
        const WaitCtl ctl{m.abort, status, 1000000000ull};
        const uint64_t ad = smem_desc_sw128(smem_u32(m.a), 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(m.b), 16, 1024);
        const uint64_t bdn = smem_desc_sw128(smem_u32(m.b), 16384, 1024);
        const long long t0 = clock64();
        for (int i = 0; i < nmma; ++i) {
            const int k = i & 3;
            if constexpr (MODE == 0)
                umma_ss(tb, desc_advance(ad, k * 32), desc_advance(bd, k * 32), idesc_bf16_f32(128, 128, false, false), i > 0);
            if constexpr (MODE == 1)
                umma_ss(tb, desc_advance(ad, k * 32), desc_advance(bd, k * 32), idesc_bf16_f32(128, 256, false, false), i > 0);
            if constexpr (MODE == 2)
                umma_ss(tb, desc_advance(ad, k * 32), desc_advance(bd, k * 32), idesc_bf16_f32(128, 64, false, false), i > 0);
            if constexpr (MODE == 3)   // A from TMEM (columns 384..447), B N-major: the P V form
                umma_ts(tb, tb + 384 + (i & 7) * 8, desc_advance(bdn, (i & 7) * 2048), idesc_bf16_f32(128, 128, false, true), i > 0);
        }
        const long long t1 = clock64();
        umma_commit(&m.bar[0]);
        mbar_wait(&m.bar[0], 0, ctl);
        const long long t2 = clock64();
        out[blockIdx.x * 2] = t1 - t0;
        out[blockIdx.x * 2 + 1] = t2 - t0;
    }
    probe_teardown(tb);
}

template <int MODE>
void run_mma(const char *name, int sms, long long *d_out, int *d_status)
{
    const int nmma = 512;
    static long long h[152 * 2];
    cudaFuncSetAttribute(mma_rate<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
    for (int rep = 0; rep < 3; ++rep) mma_rate<MODE><<<sms, 128, kProbeSmem>>>(d_out, nmma, d_status);
    const cudaError_t e = cudaDeviceSynchronize();
    int st = 0;
    cudaMemcpy(&st, d_status, 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess || st) { printf("  %s: error %s, status %d\n", name, cudaGetErrorString(e), st); return; }
    cudaMemcpy(h, d_out, sizeof(long long) * 2 * sms, cudaMemcpyDeviceToHost);
    double a = 0, b = 0;
    for (int i = 0; i < sms; ++i) { a += h[2 * i]; b += h[2 * i + 1]; }
    printf("  %-44s %6.1f cycles per MMA issued, %6.1f to completion\n", name, a / sms / nmma, b / sms / nmma);
}

// Single-thread latencies (one CTA): the thread branches on each result.
__global__ void __launch_bounds__(128, 1) sync_latency(long long *out, int *status)
{
    extern __shared__ uint8_t raw[];
    const ProbeSmem m = probe_setup(raw);
    const uint32_t tb = *m.tmem_base;
    if (threadIdx.x == 0) {
        const WaitCtl ctl{m.abort, status, 1000000000ull};
        const int N = 256;
        mbar_arrive(&m.bar[0]);   // phase 0 of barrier 0 complete
        mbar_wait(&m.bar[0], 0, ctl);
        int cnt = 0;
        long long t0 = clock64();
        for (int i = 0; i < N; ++i) cnt += mbar_wait(&m.bar[0], 0, ctl) ? 1 : 0;
        out[0] = (clock64() - t0) / N;                     // wait on a completed phase
        t0 = clock64();
        for (int i = 0; i < N; ++i) cnt += mbar_poll(smem_u32(&m.bar[0]), 0) ? 1 : 0;
        out[1] = (clock64() - t0) / N;                     // non-blocking tests, results not branched on
        t0 = clock64();
        for (int i = 0; i < N; ++i) {
            mbar_arrive(&m.bar[1]);
            mbar_wait(&m.bar[1], i & 1, ctl);
        }
        out[2] = (clock64() - t0) / N;                     // own arrive -> wait
        t0 = clock64();
        for (int i = 0; i < N; ++i) {
            umma_commit(&m.bar[2]);
            mbar_wait(&m.bar[2], i & 1, ctl);
        }
        out[3] = (clock64() - t0) / N;                     // commit with nothing pending -> seen
        const uint64_t ad = smem_desc_sw128(smem_u32(m.a), 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(m.b), 16, 1024);
        t0 = clock64();
        for (int i = 0; i < N; ++i) {
            umma_ss(tb, ad, bd, idesc_bf16_f32(128, 128, false, false), 0u);
            umma_commit(&m.bar[3]);
            mbar_wait(&m.bar[3], i & 1, ctl);
        }
        out[4] = (clock64() - t0) / N;                     // one MMA + commit -> seen
        t0 = clock64();
        for (int i = 0; i < N; ++i) {
            for (int k = 0; k < 8; ++k)
                umma_ss(tb, desc_advance(ad, (k & 3) * 32), desc_advance(bd, (k & 3) * 32),
                        idesc_bf16_f32(128, 128, false, false), k > 0);
            umma_commit(&m.bar[4]);
            mbar_wait(&m.bar[4], i & 1, ctl);
        }
        out[5] = (clock64() - t0) / N;                     // eight MMAs (one score tile) + commit -> seen
        out[6] = cnt;
    }
    probe_teardown(tb);
}

}  // namespace

int main()
{
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    if (sms > 152) sms = 152;
    float *out;
    long long *cyc, *d_out;
    int *d_status;
    cudaMalloc(&out, sizeof(float) * 152 * 512);
    cudaMalloc(&cyc, sizeof(long long) * 152 * 16);
    cudaMalloc(&d_out, sizeof(long long) * 2 * 152);
    cudaMalloc(&d_status, 4);
    cudaMemset(d_status, 0, 4);
    printf("Instruction rates (%d SMs, 512 threads each, 8 independent chains per thread):\n", sms);
    run_alu<0>("ex2.approx.ftz.f32", sms, out, cyc);
    run_alu<1>("max.f32, two inputs", sms, out, cyc);
    run_alu<2>("max.f32, three inputs", sms, out, cyc);
    run_alu<3>("fma.rn.f32", sms, out, cyc);
    run_alu<4>("add.rn.f32", sms, out, cyc);
    run_alu<5>("fma.rn.f32x2 (pairs)", sms, out, cyc);
    run_alu<6>("add.rn.f32x2 (pairs)", sms, out, cyc);
    run_alu<7>("ex2 interleaved with fma (ex2 counted)", sms, out, cyc);
    printf("tcgen05.mma kind::f16 from one thread per SM, 512 back to back (%d SMs):\n", sms);
    run_mma<0>("SS M128 N128 K16", sms, d_out, d_status);
    run_mma<1>("SS M128 N256 K16", sms, d_out, d_status);
    run_mma<2>("SS M128 N64 K16", sms, d_out, d_status);
    run_mma<3>("TS M128 N128 K16 (A in TMEM, B N-major)", sms, d_out, d_status);
    long long h[8] = {0};
    cudaFuncSetAttribute(sync_latency, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
    for (int rep = 0; rep < 2; ++rep) sync_latency<<<1, 128, kProbeSmem>>>(d_out, d_status);
    const cudaError_t e = cudaDeviceSynchronize();
    int st = 0;
    cudaMemcpy(&st, d_status, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(h, d_out, sizeof(h[0]) * 7, cudaMemcpyDeviceToHost);
    printf("Single-thread latencies (cycles; %s, status %d):\n", cudaGetErrorString(e), st);
    printf("  bounded wait on a completed mbarrier phase  %lld\n", h[0]);
    printf("  mbarrier test_wait, results not branched on  %lld\n", h[1]);
    printf("  own arrive -> wait                           %lld\n", h[2]);
    printf("  tcgen05.commit (nothing pending) -> seen      %lld\n", h[3]);
    printf("  one M128 N128 K16 MMA + commit -> seen        %lld\n", h[4]);
    printf("  eight of them + commit -> seen                %lld\n", h[5]);
    return (e == cudaSuccess && st == 0) ? 0 : 1;
}
