// ssd.cu -- Mamba-2 SSD scan (the chunk-state / chunk-scan linear-attention
// functions the TileLang paper benchmarks on H100, "TileLang: 面向AI系统的可组
// 合分块编程模型", results; the selective-scan recurrence is sketched in
// "从FlashAttention到通用内核", section 4), in its chunked form:
//   per head h (B/C group g = h / (H / G)), state S [P][N]:
//     S_t = exp(dt_t A_h) S_{t-1} + dt_t x_t B_t^T,   y_t = S_t C_t + D_h x_t.
// With a = dt A and cum the inclusive prefix sum of a inside a chunk of Q
// steps, the chunk's output is
//     y_t = sum_{s<=t} exp(cum_t - cum_s) dt_s (C_t . B_s) x_s
//           + exp(cum_t) S_in C_t + D x_t,
// and the state the chunk passes on is
//     S_out = exp(cum_end) S_in + sum_s exp(cum_end - cum_s) dt_s x_s B_s^T.
// Three kernels: the per-chunk state contributions (chunk_state), the
// sequential state passing over chunks (state_pass, in place: each chunk's
// slot ends up holding the state entering it) and the chunk outputs
// (chunk_scan).  This version runs on the CUDA cores (fp32 FFMA).
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

constexpr int kQ = 64;       // steps per chunk
constexpr int kP = 64;       // head dim
constexpr int kN = 128;      // state dim
constexpr int kThreads = 256;

struct SsdParams {
    const __nv_bfloat16 *x;   // [Bsz][L][H][P]
    const float *dt;          // [Bsz][L][H]
    const float *A;           // [H]
    const __nv_bfloat16 *Bm;  // [Bsz][L][G][N]
    const __nv_bfloat16 *Cm;  // [Bsz][L][G][N]
    const float *D;           // [H] or nullptr
    float *y;                 // [Bsz][L][H][P]
    float *S_final;           // [Bsz][H][P][N] or nullptr
    float *states;            // [Bsz][nchunks][H][P][N]
    float *dA_end;            // [Bsz][nchunks][H]: cum at the chunk's last step
    int Bsz, L, H, G, nchunks;
};

__device__ __forceinline__ float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }

// Inclusive prefix sum of a = dt * A over the chunk's steps into cum[0..len).
__device__ __forceinline__ void chunk_cumsum(const SsdParams &p, int b, int c, int h, int len, float *cum,
                                             float *dts)
{
    if (threadIdx.x < 32) {
        const float Ah = p.A[h];
        float carry = 0.f;
        for (int base = 0; base < kQ; base += 32) {
            const int s = base + threadIdx.x;
            const float d = s < len ? p.dt[(static_cast<size_t>(b) * p.L + c * kQ + s) * p.H + h] : 0.f;
            float v = d * Ah;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, v, o);
                if (threadIdx.x >= o) v += u;
            }
            cum[s] = carry + v;
            dts[s] = d;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
}

// S_c = sum_s exp(cum_end - cum_s) dt_s x_s B_s^T  ([P][N], one block per (chunk, head, batch)).
__global__ void __launch_bounds__(kThreads) ssd_chunk_state_kernel(const SsdParams p)
{
    extern __shared__ float sm[];
    float *cum = sm, *dts = sm + kQ;
    float (*xs)[kP] = reinterpret_cast<float (*)[kP]>(dts + kQ);          // x_s scaled by exp(cum_end - cum_s) dt_s
    float (*bs)[kN + 4] = reinterpret_cast<float (*)[kN + 4]>(dts + kQ + kQ * kP);
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int g = h / (p.H / p.G);
    const int len = min(kQ, p.L - c * kQ);
    chunk_cumsum(p, b, c, h, len, cum, dts);
    const float cend = cum[len - 1];
    for (int i = threadIdx.x; i < kQ * kP; i += kThreads) {
        const int s = i / kP, q = i % kP;
        float v = 0.f;
        if (s < len)
            v = bf(p.x[((static_cast<size_t>(b) * p.L + c * kQ + s) * p.H + h) * kP + q]) * __expf(cend - cum[s]) * dts[s];
        xs[s][q] = v;
    }
    for (int i = threadIdx.x; i < kQ * kN; i += kThreads) {
        const int s = i / kN, n = i % kN;
        bs[s][n] = s < len ? bf(p.Bm[((static_cast<size_t>(b) * p.L + c * kQ + s) * p.G + g) * kN + n]) : 0.f;
    }
    __syncthreads();
    // thread: rows q = ty*4 .. +4 of P, cols n = tx*8 .. +8 of N (16 x 16 threads)
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][8] = {};
    for (int s = 0; s < len; ++s) {
        float xv[4], bv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) xv[i] = xs[s][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 8; ++j) bv[j] = bs[s][tx * 8 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv[i], bv[j], acc[i][j]);
    }
    float *dst = p.states + ((static_cast<size_t>(b) * p.nchunks + c) * p.H + h) * (kP * kN);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 *o = reinterpret_cast<float4 *>(dst + (ty * 4 + i) * kN + tx * 8);
        o[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        o[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    if (threadIdx.x == 0) p.dA_end[(static_cast<size_t>(b) * p.nchunks + c) * p.H + h] = cend;
}

// In place over the chunks of each (batch, head): slot c := the state entering
// chunk c (slot 0 := 0), from the chunk contributions and exp(cum_end).  One
// thread per state element.
__global__ void __launch_bounds__(kThreads) ssd_state_pass_kernel(const SsdParams p)
{
    const int e = blockIdx.x * kThreads + threadIdx.x;      // element of [P][N]
    const int h = blockIdx.y, b = blockIdx.z;
    float carry = 0.f;
    for (int c = 0; c < p.nchunks; ++c) {
        float *slot = p.states + ((static_cast<size_t>(b) * p.nchunks + c) * p.H + h) * (kP * kN) + e;
        const float contrib = *slot;
        *slot = carry;
        carry = __expf(p.dA_end[(static_cast<size_t>(b) * p.nchunks + c) * p.H + h]) * carry + contrib;
    }
    if (p.S_final) p.S_final[(static_cast<size_t>(b) * p.H + h) * (kP * kN) + e] = carry;
}

// y of one chunk: intra-chunk products, the entering state, and D x.
__global__ void __launch_bounds__(kThreads) ssd_chunk_scan_kernel(const SsdParams p)
{
    extern __shared__ float sm[];
    float *cum = sm;                        // [Q]
    float *dts = cum + kQ;                  // [Q]
    float *cs = dts + kQ;                   // [Q][N + 4]
    float *bs = cs + kQ * (kN + 4);         // [Q][N + 4]
    float *w = bs + kQ * (kN + 4);          // [Q][Q + 4]: exp(cum_t - cum_s) dt_s (C_t . B_s), s <= t
    float *xs = w + kQ * (kQ + 4);          // [Q][P]
    float *st = xs + kQ * kP;               // [P][N + 4]: the entering state
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int g = h / (p.H / p.G);
    const int len = min(kQ, p.L - c * kQ);
    chunk_cumsum(p, b, c, h, len, cum, dts);
    for (int i = threadIdx.x; i < kQ * kN; i += kThreads) {
        const int s = i / kN, n = i % kN;
        const size_t src = ((static_cast<size_t>(b) * p.L + c * kQ + s) * p.G + g) * kN + n;
        cs[s * (kN + 4) + n] = s < len ? bf(p.Cm[src]) : 0.f;
        bs[s * (kN + 4) + n] = s < len ? bf(p.Bm[src]) : 0.f;
    }
    for (int i = threadIdx.x; i < kQ * kP; i += kThreads) {
        const int s = i / kP, q = i % kP;
        xs[i] = s < len ? bf(p.x[((static_cast<size_t>(b) * p.L + c * kQ + s) * p.H + h) * kP + q]) : 0.f;
    }
    const float *S_in = p.states + ((static_cast<size_t>(b) * p.nchunks + c) * p.H + h) * (kP * kN);
    for (int i = threadIdx.x; i < kP * kN; i += kThreads) st[(i / kN) * (kN + 4) + i % kN] = S_in[i];
    __syncthreads();
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    // W[t][s] for t = ty*4..+4, s = tx*4..+4
    {
        float acc[4][4] = {};
        for (int n = 0; n < kN; ++n) {
            float cv[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cv[i] = cs[(ty * 4 + i) * (kN + 4) + n];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = bs[(tx * 4 + j) * (kN + 4) + n];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(cv[i], bv[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = ty * 4 + i, s = tx * 4 + j;
                w[t * (kQ + 4) + s] = (s <= t && t < len) ? acc[i][j] * __expf(cum[t] - cum[s]) * dts[s] : 0.f;
            }
    }
    __syncthreads();
    // y[t][q] for t = ty*4..+4, q = tx*4..+4
    float acc[4][4] = {};
    for (int s = 0; s < kQ; ++s) {
        float wv[4], xv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wv[i] = w[(ty * 4 + i) * (kQ + 4) + s];
#pragma unroll
        for (int j = 0; j < 4; ++j) xv[j] = xs[s * kP + tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(wv[i], xv[j], acc[i][j]);
    }
    float acc2[4][4] = {};
    for (int n = 0; n < kN; ++n) {
        float cv[4], sv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) cv[i] = cs[(ty * 4 + i) * (kN + 4) + n];
#pragma unroll
        for (int j = 0; j < 4; ++j) sv[j] = st[(tx * 4 + j) * (kN + 4) + n];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc2[i][j] = fmaf(cv[i], sv[j], acc2[i][j]);
    }
    const float Dh = p.D ? p.D[h] : 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = ty * 4 + i;
        if (t >= len) continue;
        const float e = __expf(cum[t]);
        float out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j] = acc[i][j] + e * acc2[i][j] + Dh * xs[t * kP + tx * 4 + j];
        float4 *dst = reinterpret_cast<float4 *>(p.y + ((static_cast<size_t>(b) * p.L + c * kQ + t) * p.H + h) * kP +
                                                 tx * 4);
        *dst = make_float4(out[0], out[1], out[2], out[3]);
    }
}

constexpr size_t kStateSmem = sizeof(float) * (2 * kQ + kQ * kP + kQ * (kN + 4));
constexpr size_t kScanSmem =
    sizeof(float) * (2 * kQ + 2 * kQ * (kN + 4) + kQ * (kQ + 4) + kQ * kP + kP * (kN + 4));

}  // namespace

size_t ssd_workspace_bytes(int Bsz, int L, int H)
{
    const size_t nchunks = (static_cast<size_t>(L) + kQ - 1) / kQ;
    return nchunks * Bsz * H * (static_cast<size_t>(kP) * kN + 1) * sizeof(float);
}

int launch_ssd_scan(const void *x, const float *dt, const float *A, const void *Bm, const void *Cm, const float *D,
                    float *y, float *S_final, int Bsz, int L, int H, int P, int G, int N, void *workspace,
                    size_t workspace_bytes, const LaunchEnv &env, std::string &err)
{
    if (P != kP || N != kN) {
        err = "ssd_scan: supports P = 64, N = 128";
        return 2;
    }
    if (workspace_bytes < ssd_workspace_bytes(Bsz, L, H)) {
        err = "ssd_scan: workspace too small";
        return 4;
    }
    SsdParams p;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.dt = dt;
    p.A = A;
    p.Bm = static_cast<const __nv_bfloat16 *>(Bm);
    p.Cm = static_cast<const __nv_bfloat16 *>(Cm);
    p.D = D;
    p.y = y;
    p.S_final = S_final;
    p.Bsz = Bsz;
    p.L = L;
    p.H = H;
    p.G = G;
    p.nchunks = (L + kQ - 1) / kQ;
    p.states = static_cast<float *>(workspace);
    p.dA_end = p.states + static_cast<size_t>(p.nchunks) * Bsz * H * kP * kN;
    const dim3 grid(p.nchunks, H, Bsz);
    static bool configured = false;
    cudaError_t e = cudaSuccess;
    if (!configured) {
        e = cudaFuncSetAttribute(ssd_chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kStateSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ssd_chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kScanSmem));
        configured = e == cudaSuccess;
    }
    if (e == cudaSuccess) {
        ssd_chunk_state_kernel<<<grid, kThreads, kStateSmem, env.stream>>>(p);
        ssd_state_pass_kernel<<<dim3(kP * kN / kThreads, H, Bsz), kThreads, 0, env.stream>>>(p);
        ssd_chunk_scan_kernel<<<grid, kThreads, kScanSmem, env.stream>>>(p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        err = std::string("ssd_scan launch: ") + cudaGetErrorString(e);
        return 5;
    }
    return 0;
}

}  // namespace gbattn
