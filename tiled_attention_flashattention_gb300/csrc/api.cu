// api.cu -- the C ABI of libgbattn.so (declared in include/gbattn.h):
// argument validation, per-device state (architecture check, SM count, device
// status word), TMA descriptor encoding, and dispatch to the kernel launchers.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>
#include <unordered_map>
#include <algorithm>

#include "gbattn.h"
#include "kernels.h"

namespace gbattn {
namespace {

thread_local std::string g_err;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_inject{0};

// Device status word: kernels record the first failed bounded wait here.
__device__ int g_status_word;

struct DevInfo {
    bool init = false;
    int major = 0, minor = 0, num_sms = 0;
    int *status = nullptr;
};
std::mutex g_mu;
DevInfo g_dev[64];

int fail(int code, const std::string &msg)
{
    g_err = msg;
    return code;
}

int get_env(LaunchEnv &env, void *stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(GBATTN_ERR_LAUNCH, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(GBATTN_ERR_LAUNCH, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &d = g_dev[dev];
    if (!d.init) {
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail(GBATTN_ERR_LAUNCH, std::string("device query: ") + cudaGetErrorString(e));
        if (d.major == 10 && d.minor == 3) {
            if ((e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_status_word)) != cudaSuccess)
                return fail(GBATTN_ERR_LAUNCH, std::string("status word: ") + cudaGetErrorString(e));
        }
        d.init = true;
    }
    if (!(d.major == 10 && d.minor == 3)) {
        char buf[96];
        snprintf(buf, sizeof buf, "device is sm_%d%d; this library is built for sm_103a only", d.major, d.minor);
        return fail(GBATTN_ERR_ARCH, buf);
    }
    env.stream = static_cast<cudaStream_t>(stream);
    env.status = d.status;
    env.timeout_ns = g_timeout_ns.load();
    env.num_sms = d.num_sms;
    env.inject = g_inject.load();
    return GBATTN_OK;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool valid_scale(float s)
{
    return std::isfinite(s) && s > 0.f;
}

}  // namespace

namespace {
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn tensor_map_encoder()
{
    static EncodeFn encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<EncodeFn>(fn);
    });
    return encode;
}

// Tensor maps are a pure function of their parameters, so encoded maps are
// cached by value (base address, type, dims, strides, box): repeated calls on
// the same buffers skip the driver's encode.  Bounded; cleared when full.
struct MapKey {
    uintptr_t base;
    int dtype, rank, swizzle;
    uint64_t dims[5], strides[4];
    uint32_t box[5];
    bool operator==(const MapKey &o) const
    {
        return base == o.base && dtype == o.dtype && rank == o.rank && swizzle == o.swizzle &&
               std::equal(dims, dims + 5, o.dims) &&
               std::equal(strides, strides + 4, o.strides) && std::equal(box, box + 5, o.box);
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const
    {
        uint64_t h = 1469598103934665603ull;
        auto mix = [&](uint64_t v) { h = (h ^ v) * 1099511628211ull; };
        mix(k.base);
        mix(static_cast<uint64_t>(k.dtype) << 16 | static_cast<uint64_t>(k.rank) << 8 |
            static_cast<uint64_t>(k.swizzle));
        for (uint64_t v : k.dims) mix(v);
        for (uint64_t v : k.strides) mix(v);
        for (uint32_t v : k.box) mix(v);
        return static_cast<size_t>(h);
    }
};
constexpr size_t kMapCacheMax = 1024;
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

// Encode (or fetch) a tiled map (128-byte swizzle unless given); rank <= 5.
CUresult encode_cached(CUtensorMap &desc, CUtensorMapDataType dtype, int rank, const void *base,
                       const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                       CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    MapKey key{};
    key.base = reinterpret_cast<uintptr_t>(base);
    key.dtype = static_cast<int>(dtype);
    key.rank = rank;
    key.swizzle = static_cast<int>(swizzle);
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides[i];
    }
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            desc = it->second;
            return CUDA_SUCCESS;
        }
    }
    EncodeFn encode = tensor_map_encoder();
    if (!encode) return CUDA_ERROR_NOT_SUPPORTED;
    const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    CUresult r = encode(&desc, dtype, static_cast<cuuint32_t>(rank), const_cast<void *>(base), dims, strides, box,
                        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lk(g_map_mu);
        if (g_maps.size() >= kMapCacheMax) g_maps.clear();
        g_maps.emplace(key, desc);
    }
    return r;
}
}  // namespace

bool make_tma_bf16_3d(CUtensorMap &desc, const void *base, uint64_t cols, uint64_t rows,
                      uint64_t outer, uint32_t box_rows, std::string &err)
{
    if (!tensor_map_encoder()) {
        err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    const cuuint64_t dims[3] = {cols, rows, outer};
    const cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    CUresult r = encode_cached(desc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for [%llu,%llu,%llu] box rows %u",
                 static_cast<int>(r), static_cast<unsigned long long>(outer),
                 static_cast<unsigned long long>(rows), static_cast<unsigned long long>(cols), box_rows);
        err = buf;
        return false;
    }
    return true;
}

bool make_tma_bf16_3d_sw64(CUtensorMap &desc, const void *base, uint64_t cols, uint64_t rows, uint64_t outer,
                           uint32_t box_rows, std::string &err)
{
    if (!tensor_map_encoder()) {
        err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    const cuuint64_t dims[3] = {cols, rows, outer};
    const cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
    const cuuint32_t box[3] = {32, box_rows, 1};
    CUresult r = encode_cached(desc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_64B);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for a 64-byte-swizzled [%llu,%llu,%llu] map",
                 static_cast<int>(r), static_cast<unsigned long long>(outer), static_cast<unsigned long long>(rows),
                 static_cast<unsigned long long>(cols));
        err = buf;
        return false;
    }
    return true;
}

bool make_tma_bf16_chunked(CUtensorMap &desc, const void *base, uint64_t cols, uint64_t rows, uint64_t outer,
                           uint32_t box_rows, uint32_t box_chunks, std::string &err)
{
    if (!tensor_map_encoder()) {
        err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    // [outer][rows][cols] viewed as (64 columns, rows, cols / 64 chunks, outer):
    // the chunk index is outside the row index in the box, so a box lands in
    // shared memory as [chunk][row][64 columns].
    const cuuint64_t dims[4] = {64, rows, cols / 64, outer};
    const cuuint64_t strides[3] = {cols * 2, 128, cols * rows * 2};
    const cuuint32_t box[4] = {64, box_rows, box_chunks, 1};
    CUresult r = encode_cached(desc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box);
    if (r != CUDA_SUCCESS) {
        char buf[200];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for chunked [%llu,%llu,%llu] box %u rows x %u chunks",
                 static_cast<int>(r), static_cast<unsigned long long>(outer), static_cast<unsigned long long>(rows),
                 static_cast<unsigned long long>(cols), box_rows, box_chunks);
        err = buf;
        return false;
    }
    return true;
}

bool make_tma_5d(CUtensorMap &desc, const void *base, const uint64_t (&dims)[5], const uint64_t (&strides)[4],
                 const uint32_t (&box)[5], std::string &err)
{
    if (!tensor_map_encoder()) {
        err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    const cuuint64_t d[5] = {dims[0], dims[1], dims[2], dims[3], dims[4]};
    const cuuint64_t st[4] = {strides[0], strides[1], strides[2], strides[3]};
    const cuuint32_t bx[5] = {box[0], box[1], box[2], box[3], box[4]};
    CUresult r = encode_cached(desc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, d, st, bx);
    if (r != CUDA_SUCCESS) {
        char buf[160];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for a 5-d bf16 map", static_cast<int>(r));
        err = buf;
        return false;
    }
    return true;
}

bool make_tma_4d(CUtensorMap &desc, bool f32, const void *base, const uint64_t (&dims)[4],
                 const uint64_t (&strides)[3], const uint32_t (&box)[4], std::string &err)
{
    if (!tensor_map_encoder()) {
        err = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
    const cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
    const cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
    CUresult r = encode_cached(desc, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                               base, d, st, bx);
    if (r != CUDA_SUCCESS) {
        char buf[200];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d) for dims [%llu,%llu,%llu,%llu]",
                 static_cast<int>(r), static_cast<unsigned long long>(dims[3]),
                 static_cast<unsigned long long>(dims[2]), static_cast<unsigned long long>(dims[1]),
                 static_cast<unsigned long long>(dims[0]));
        err = buf;
        return false;
    }
    return true;
}

}  // namespace gbattn

using namespace gbattn;

static int attn_fwd_common(const char *name, const void *Q, const void *K, const void *V, void *O, float *LSE,
                           const uint8_t *block_mask, bool sparse, int B, int H, int H_kv, int N_q, int N_kv,
                           int d, int causal, int window, float scale, void *stream)
{
    g_err.clear();
    const std::string n(name);
    if (B < 0 || H < 1 || H_kv < 1 || N_q < 0 || N_kv < 0)
        return fail(GBATTN_ERR_INVALID_ARG, n + ": need B >= 0, H >= 1, H_kv >= 1, N_q >= 0, N_kv >= 0");
    if (H % H_kv != 0) return fail(GBATTN_ERR_INVALID_ARG, n + ": H must be a multiple of H_kv");
    if (causal != 0 && causal != 1) return fail(GBATTN_ERR_INVALID_ARG, n + ": causal must be 0 or 1");
    if (!valid_scale(scale)) return fail(GBATTN_ERR_INVALID_ARG, n + ": scale must be finite and > 0");
    if (d != 64 && d != 128) return fail(GBATTN_ERR_UNSUPPORTED, n + ": d must be 64 or 128");
    if (static_cast<long long>(B) * H * N_q > (1LL << 40) || static_cast<long long>(N_q) * d > (1LL << 31) ||
        static_cast<long long>(N_kv) * d > (1LL << 31))
        return fail(GBATTN_ERR_UNSUPPORTED, n + ": problem too large");
    const bool work = static_cast<long long>(B) * H * N_q > 0;
    if (work && (!Q || !O || !LSE || (N_kv > 0 && (!K || !V)) || (sparse && N_kv > 0 && !block_mask)))
        return fail(GBATTN_ERR_INVALID_ARG, n + ": null tensor pointer");
    if (work && (!aligned16(Q) || !aligned16(O) || (N_kv > 0 && (!aligned16(K) || !aligned16(V)))))
        return fail(GBATTN_ERR_ALIGNMENT, n + ": Q, K, V and O must be 16-byte aligned");
    if (work && (reinterpret_cast<uintptr_t>(LSE) & 3u))
        return fail(GBATTN_ERR_ALIGNMENT, n + ": LSE must be 4-byte aligned");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    if (!work) return GBATTN_OK;
    std::string err;
    rc = launch_attn_fwd(Q, K, V, O, LSE, B, H, H_kv, N_q, N_kv, d, causal, window, scale,
                         sparse ? block_mask : nullptr, env, err);
    if (rc != GBATTN_OK) g_err = err;
    return rc;
}

extern "C" int attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                        int H_kv, int N_q, int N_kv, int d, int causal, int window, float scale,
                        void *stream)
{
    return attn_fwd_common("attn_fwd", Q, K, V, O, LSE, nullptr, false, B, H, H_kv, N_q, N_kv, d, causal, window,
                           scale, stream);
}

extern "C" int attn_fwd_sparse(const void *Q, const void *K, const void *V, void *O, float *LSE,
                               const unsigned char *block_mask, int B, int H, int H_kv, int N_q, int N_kv, int d,
                               int causal, int window, float scale, void *stream)
{
    return attn_fwd_common("attn_fwd_sparse", Q, K, V, O, LSE, block_mask, true, B, H, H_kv, N_q, N_kv, d, causal,
                           window, scale, stream);
}

extern "C" size_t mla_decode_workspace_bytes(int B, int H, int N_kv, int d_c)
{
    if (B < 1 || H < 1 || N_kv < 1 || d_c < 1) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return mla_workspace_bytes(B, H, N_kv, d_c, sms);
}

extern "C" int mla_decode(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe,
                          void *O, float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    g_err.clear();
    if (B < 1 || H < 1 || N_kv < 1 || d_c < 1 || d_r < 0)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode: need B, H, N_kv, d_c >= 1 and d_r >= 0");
    if (!valid_scale(scale)) return fail(GBATTN_ERR_INVALID_ARG, "mla_decode: scale must be finite and > 0");
    if (d_c != 512 || d_r != 64 || H > 128)
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode: supports d_c = 512, d_r = 64, H <= 128");
    if (static_cast<long long>(N_kv) * d_c > (1LL << 31))
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode: problem too large");
    if (!Q_nope || !Q_pe || !KV_latent || !K_pe || !O || !LSE)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode: null tensor pointer");
    if (!aligned16(Q_nope) || !aligned16(Q_pe) || !aligned16(KV_latent) || !aligned16(K_pe) || !aligned16(O) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u))
        return fail(GBATTN_ERR_ALIGNMENT, "mla_decode: tensors must be 16-byte aligned (LSE 4-byte)");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    const size_t need = mla_workspace_bytes(B, H, N_kv, d_c, env.num_sms);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return fail(GBATTN_ERR_WORKSPACE, "mla_decode: workspace missing, smaller than "
                                          "mla_decode_workspace_bytes() or not 16-byte aligned");
    std::string err;
    rc = launch_mla_decode(Q_nope, Q_pe, KV_latent, K_pe, O, LSE, B, H, N_kv, d_c, d_r, scale,
                           workspace, workspace_bytes, env, err);
    if (rc != GBATTN_OK) g_err = err;
    return rc;
}

extern "C" int mla_decode_noalloc(const void *Q_nope, const void *Q_pe, const void *KV_latent,
                                  const void *K_pe, void *O, float *LSE, int B, int H, int N_kv, int d_c,
                                  int d_r, float scale, void *stream)
{
    g_err.clear();
    if (B < 1 || H < 1 || N_kv < 1 || d_c < 1 || d_r < 0)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_noalloc: need B, H, N_kv, d_c >= 1 and d_r >= 0");
    if (!valid_scale(scale))
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_noalloc: scale must be finite and > 0");
    if (d_c != 512 || d_r != 64 || H > 128)
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode_noalloc: supports d_c = 512, d_r = 64, H <= 128");
    if (static_cast<long long>(N_kv) * d_c > (1LL << 31))
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode_noalloc: problem too large");
    if (!Q_nope || !Q_pe || !KV_latent || !K_pe || !O || !LSE)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_noalloc: null tensor pointer");
    if (!aligned16(Q_nope) || !aligned16(Q_pe) || !aligned16(KV_latent) || !aligned16(K_pe) || !aligned16(O) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u))
        return fail(GBATTN_ERR_ALIGNMENT, "mla_decode_noalloc: tensors must be 16-byte aligned (LSE 4-byte)");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    std::string err;
    rc = launch_mla_decode_noalloc(Q_nope, Q_pe, KV_latent, K_pe, O, LSE, B, H, N_kv, d_c, d_r, scale, env, err);
    if (rc != GBATTN_OK) g_err = err;
    return rc;
}

extern "C" size_t mla_decode_paged_workspace_bytes(int B, int s_q, int H, int d_c)
{
    if (B < 1 || s_q < 1 || H < 1 || d_c < 1) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return mla_paged_workspace_bytes(B, s_q, H, d_c, sms);
}

extern "C" int mla_decode_paged(const void *Q_nope, const void *Q_pe, const void *KV_cache, const void *K_pe_cache,
                                const int *block_table, const int *cache_seqlens, void *O, float *LSE, int B, int s_q,
                                int H, int num_pages, int max_pages_per_seq, int page_size, int d_c, int d_r,
                                float scale, void *workspace, size_t workspace_bytes, void *stream)
{
    g_err.clear();
    if (B < 1 || s_q < 1 || H < 1 || num_pages < 1 || max_pages_per_seq < 1 || d_c < 1 || d_r < 0 || page_size < 1)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_paged: need B, s_q, H, num_pages, max_pages_per_seq, d_c, "
                                            "page_size >= 1 and d_r >= 0");
    if (!valid_scale(scale)) return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_paged: scale must be finite and > 0");
    if (d_c != 512 || d_r != 64 || H > 128 || page_size != 64)
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode_paged: supports d_c = 512, d_r = 64, H <= 128, page_size = 64");
    if (static_cast<long long>(B) * s_q * max_pages_per_seq > 0x7fffffffLL ||
        static_cast<long long>(max_pages_per_seq) * page_size > 0x7fffffffLL)
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode_paged: problem too large");
    if (!Q_nope || !Q_pe || !KV_cache || !K_pe_cache || !block_table || !cache_seqlens || !O || !LSE)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_paged: null pointer");
    if (!aligned16(Q_nope) || !aligned16(Q_pe) || !aligned16(KV_cache) || !aligned16(K_pe_cache) || !aligned16(O) ||
        (reinterpret_cast<uintptr_t>(LSE) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u))
        return fail(GBATTN_ERR_ALIGNMENT, "mla_decode_paged: tensors must be 16-byte aligned "
                                          "(LSE, block_table, cache_seqlens 4-byte)");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    const size_t need = mla_paged_workspace_bytes(B, s_q, H, d_c, env.num_sms);
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(GBATTN_ERR_WORKSPACE, "mla_decode_paged: workspace missing, smaller than "
                                          "mla_decode_paged_workspace_bytes() or not 16-byte aligned");
    std::string err;
    rc = launch_mla_decode_paged(Q_nope, Q_pe, KV_cache, K_pe_cache, block_table, cache_seqlens, O, LSE, B, s_q, H,
                                 num_pages, max_pages_per_seq, d_c, d_r, scale, workspace, workspace_bytes, env,
                                 err);
    if (rc != GBATTN_OK) g_err = err;
    return rc;
}

extern "C" int ssd_scan(const void *x, const float *dt, const float *A, const void *B, const void *C, const float *D,
                        float *y, float *final_state, int Bsz, int L, int H, int P, int G, int N, void *stream)
{
    g_err.clear();
    if (Bsz < 1 || L < 1 || H < 1 || G < 1 || P < 1 || N < 1)
        return fail(GBATTN_ERR_INVALID_ARG, "ssd_scan: need Bsz, L, H, G, P, N >= 1");
    if (H % G != 0) return fail(GBATTN_ERR_INVALID_ARG, "ssd_scan: H must be a multiple of G");
    if (P != 64 || N != 128) return fail(GBATTN_ERR_UNSUPPORTED, "ssd_scan: supports P = 64, N = 128");
    if (Bsz > 65535) return fail(GBATTN_ERR_UNSUPPORTED, "ssd_scan: Bsz > 65535");
    if (!x || !dt || !A || !B || !C || !y)
        return fail(GBATTN_ERR_INVALID_ARG, "ssd_scan: null tensor pointer");
    auto al4 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
    if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(y) ||
        (final_state && !aligned16(final_state)) || !al4(dt) || !al4(A) || (D && !al4(D)))
        return fail(GBATTN_ERR_ALIGNMENT, "ssd_scan: x, B, C, y, final_state must be 16-byte aligned "
                                          "(dt, A, D 4-byte)");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    std::string err;
    rc = launch_ssd_scan(x, dt, A, B, C, D, y, final_state, Bsz, L, H, P, G, N, env, err);
    if (rc != GBATTN_OK) g_err = err;
    return rc;
}

// ---------------------------------------------------------------------------
// Host-buffer entry points: the same computation with inputs and outputs in
// host memory.  The work is cut into a few contiguous chunks of (batch,
// KV-head) units (each a valid problem on sub-tensors), and per chunk the
// host-to-device copies (two helper streams, two copy engines), the kernels
// and the device-to-host copies (a third helper stream) are chained by events,
// so the copies of one chunk overlap the kernels and copies of the others.
// attn_fwd_host runs the chunks' kernels on two more helper streams, so that
// one chunk's kernel starts while the previous one's last CTAs finish;
// mla_decode_host runs them on the caller's stream (the chunks share one
// split-KV workspace).  Pinned host memory gives asynchronous copies; pageable
// memory works but copies synchronously.

namespace {
constexpr int kPipeChunks = 8;          // events per helper stream (the most chunks of any call)
constexpr int kAttnChunks = 8;          // attn_fwd_host: chunks of (batch, KV-head) units
constexpr int kMlaChunks = 4;           // mla_decode_host: chunks of sequences (fewer sequences per
                                        // launch make the split-KV plan split more)

struct HostPipe {
    std::mutex mu;            // held while a call enqueues (events are reused)
    bool init = false;
    cudaStream_t h2d[2] = {nullptr, nullptr}, d2h = nullptr;   // two copy-in streams: two copy engines
    cudaStream_t kern[2] = {nullptr, nullptr};                 // attn_fwd_host's chunk kernels
    cudaEvent_t start = nullptr;
    cudaEvent_t ev_in[2][kPipeChunks], ev_k[kPipeChunks], ev_out = nullptr;
};
HostPipe g_pipe[64];

int host_pipe(HostPipe *&hp)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) return fail(GBATTN_ERR_LAUNCH, "host pipeline: no device");
    hp = &g_pipe[dev];
    static std::mutex init_mu;
    std::lock_guard<std::mutex> lk(init_mu);
    if (hp->init) return GBATTN_OK;
    const unsigned ef = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&hp->h2d[0], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->h2d[1], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->kern[0], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->kern[1], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->start, ef);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->ev_out, ef);
    for (int i = 0; i < kPipeChunks && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&hp->ev_in[0][i], ef);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->ev_in[1][i], ef);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp->ev_k[i], ef);
    }
    if (e != cudaSuccess) return fail(GBATTN_ERR_LAUNCH, std::string("host pipeline setup: ") + cudaGetErrorString(e));
    hp->init = true;
    return GBATTN_OK;
}

size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// One host-to-device or device-to-host piece of a chunk.
struct Piece {
    void *dst;
    const void *src;
    size_t bytes;
};

// The helper streams start after what the caller queued on `user`.
cudaError_t pipe_start(HostPipe *hp, cudaStream_t user)
{
    cudaError_t e = cudaEventRecord(hp->start, user);
    for (int j = 0; j < 2 && e == cudaSuccess; ++j) e = cudaStreamWaitEvent(hp->h2d[j], hp->start, 0);
    for (int j = 0; j < 2 && e == cudaSuccess; ++j) e = cudaStreamWaitEvent(hp->kern[j], hp->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->start, 0);
    return e;
}

// Copy a chunk's inputs in, alternating pieces between the two copy-in
// streams, and make `user` wait for both.
template <int N>
cudaError_t pipe_copy_in(HostPipe *hp, int c, const Piece (&in)[N], cudaStream_t user)
{
    cudaError_t e = cudaSuccess;
    int j = 0;
    for (const Piece &pc : in)
        if (e == cudaSuccess && pc.bytes) {
            e = cudaMemcpyAsync(pc.dst, pc.src, pc.bytes, cudaMemcpyHostToDevice, hp->h2d[j]);
            j ^= 1;
        }
    for (int s = 0; s < 2 && e == cudaSuccess; ++s) {
        e = cudaEventRecord(hp->ev_in[s][c], hp->h2d[s]);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(user, hp->ev_in[s][c], 0);
    }
    return e;
}
}  // namespace

extern "C" size_t attn_fwd_host_device_bytes(int B, int H, int H_kv, int N_q, int N_kv, int d)
{
    if (B < 1 || H < 1 || H_kv < 1 || N_q < 0 || N_kv < 0 || d < 1) return 0;
    const size_t q = static_cast<size_t>(B) * H * N_q * d * 2, kv = static_cast<size_t>(B) * H_kv * N_kv * d * 2;
    return 2 * round256(q) + 2 * round256(kv) + round256(static_cast<size_t>(B) * H * N_q * 4);
}

extern "C" int attn_fwd_host(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                             int H_kv, int N_q, int N_kv, int d, int causal, int window, float scale,
                             void *device_buf, size_t device_bytes, void *stream)
{
    g_err.clear();
    if (B < 1 || H < 1 || H_kv < 1 || N_q < 0 || N_kv < 0)
        return fail(GBATTN_ERR_INVALID_ARG, "attn_fwd_host: need B, H, H_kv >= 1, N_q, N_kv >= 0");
    if (H % H_kv != 0) return fail(GBATTN_ERR_INVALID_ARG, "attn_fwd_host: H must be a multiple of H_kv");
    if (causal != 0 && causal != 1) return fail(GBATTN_ERR_INVALID_ARG, "attn_fwd_host: causal must be 0 or 1");
    if (!valid_scale(scale)) return fail(GBATTN_ERR_INVALID_ARG, "attn_fwd_host: scale must be finite and > 0");
    if (d != 64 && d != 128) return fail(GBATTN_ERR_UNSUPPORTED, "attn_fwd_host: d must be 64 or 128");
    if (static_cast<long long>(B) * H * N_q > (1LL << 40) || static_cast<long long>(N_q) * d > (1LL << 31) ||
        static_cast<long long>(N_kv) * d > (1LL << 31))
        return fail(GBATTN_ERR_UNSUPPORTED, "attn_fwd_host: problem too large");
    if (N_q == 0) return GBATTN_OK;
    if (!Q || !O || !LSE || (N_kv > 0 && (!K || !V)))
        return fail(GBATTN_ERR_INVALID_ARG, "attn_fwd_host: null tensor pointer");
    const size_t need = attn_fwd_host_device_bytes(B, H, H_kv, N_q, N_kv, d);
    if (!device_buf || device_bytes < need || (reinterpret_cast<uintptr_t>(device_buf) & 255u))
        return fail(GBATTN_ERR_WORKSPACE, "attn_fwd_host: device buffer missing, smaller than "
                                          "attn_fwd_host_device_bytes() or not 256-byte aligned");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    HostPipe *hp = nullptr;
    if ((rc = host_pipe(hp)) != GBATTN_OK) return rc;
    std::lock_guard<std::mutex> lk(hp->mu);

    const size_t qb = static_cast<size_t>(B) * H * N_q * d * 2, kvb = static_cast<size_t>(B) * H_kv * N_kv * d * 2;
    uint8_t *dQ = static_cast<uint8_t *>(device_buf), *dK = dQ + round256(qb), *dV = dK + round256(kvb),
            *dO = dV + round256(kvb), *dL = dO + round256(qb);
    const int group = H / H_kv, units = B * H_kv;
    const int nchunk = std::min(kAttnChunks, units);
    const size_t q_unit = static_cast<size_t>(group) * N_q * d * 2, kv_unit = static_cast<size_t>(N_kv) * d * 2,
                 l_unit = static_cast<size_t>(group) * N_q * 4;
    cudaError_t e = pipe_start(hp, env.stream);
    std::string err;
    for (int c = 0; c < nchunk && e == cudaSuccess; ++c) {
        const int u0 = static_cast<int>(static_cast<long long>(c) * units / nchunk);
        const int u1 = static_cast<int>(static_cast<long long>(c + 1) * units / nchunk);
        const int nu = u1 - u0;
        const Piece in[3] = {{dQ + u0 * q_unit, static_cast<const uint8_t *>(Q) + u0 * q_unit, nu * q_unit},
                             {dK + u0 * kv_unit, K ? static_cast<const uint8_t *>(K) + u0 * kv_unit : nullptr,
                              nu * kv_unit},
                             {dV + u0 * kv_unit, V ? static_cast<const uint8_t *>(V) + u0 * kv_unit : nullptr,
                              nu * kv_unit}};
        // this chunk's kernel on helper stream c % 2: it can start while the
        // previous chunk's kernel drains on the other one
        LaunchEnv kenv = env;
        kenv.stream = hp->kern[c & 1];
        e = pipe_copy_in(hp, c, in, kenv.stream);
        if (e != cudaSuccess) break;
        rc = launch_attn_fwd(dQ + u0 * q_unit, dK + u0 * kv_unit, dV + u0 * kv_unit, dO + u0 * q_unit,
                             reinterpret_cast<float *>(dL + u0 * l_unit), 1, nu * group, nu, N_q, N_kv, d, causal,
                             window, scale, nullptr, kenv, err);
        if (rc != GBATTN_OK) {
            g_err = err;
            return rc;
        }
        e = cudaEventRecord(hp->ev_k[c], kenv.stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->ev_k[c], 0);
        const Piece out[2] = {{static_cast<uint8_t *>(O) + u0 * q_unit, dO + u0 * q_unit, nu * q_unit},
                              {reinterpret_cast<uint8_t *>(LSE) + u0 * l_unit, dL + u0 * l_unit, nu * l_unit}};
        for (const Piece &pc : out)
            if (e == cudaSuccess) e = cudaMemcpyAsync(pc.dst, pc.src, pc.bytes, cudaMemcpyDeviceToHost, hp->d2h);
    }
    // the caller's stream continues once the last copy back is done (every
    // chunk's copy back waited for that chunk's kernel)
    if (e == cudaSuccess) e = cudaEventRecord(hp->ev_out, hp->d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(env.stream, hp->ev_out, 0);
    if (e != cudaSuccess) return fail(GBATTN_ERR_LAUNCH, std::string("attn_fwd_host: ") + cudaGetErrorString(e));
    return GBATTN_OK;
}

// Split-KV workspace for the chunks of a host-buffer MLA call: the largest plan
// over the chunk sizes (the plan depends on the number of sequences).
static size_t mla_host_chunk_workspace(int B, int H, int N_kv, int d_c, int num_sms)
{
    const int n = std::min(kMlaChunks, B);
    size_t ws = 0;
    for (int c = 0; c < n; ++c) {
        const int nb = static_cast<int>(static_cast<long long>(c + 1) * B / n - static_cast<long long>(c) * B / n);
        ws = std::max(ws, mla_workspace_bytes(nb, H, N_kv, d_c, num_sms));
    }
    return ws;
}

extern "C" size_t mla_decode_host_device_bytes(int B, int H, int N_kv, int d_c, int d_r)
{
    if (B < 1 || H < 1 || N_kv < 1 || d_c < 1 || d_r < 0) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 0;
    const size_t ws = sms > 0 ? mla_host_chunk_workspace(B, H, N_kv, d_c, sms) : 0;
    const size_t b = static_cast<size_t>(B);
    return round256(b * H * d_c * 2) + round256(b * H * d_r * 2) + round256(b * N_kv * d_c * 2) +
           round256(b * N_kv * d_r * 2) + round256(b * H * d_c * 2) + round256(b * H * 4) + round256(ws);
}

extern "C" int mla_decode_host(const void *Q_nope, const void *Q_pe, const void *KV_latent, const void *K_pe,
                               void *O, float *LSE, int B, int H, int N_kv, int d_c, int d_r, float scale,
                               void *device_buf, size_t device_bytes, void *stream)
{
    g_err.clear();
    if (B < 1 || H < 1 || N_kv < 1 || d_c < 1 || d_r < 0)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_host: need B, H, N_kv, d_c >= 1 and d_r >= 0");
    if (!valid_scale(scale)) return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_host: scale must be finite and > 0");
    if (d_c != 512 || d_r != 64 || H > 128)
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode_host: supports d_c = 512, d_r = 64, H <= 128");
    if (static_cast<long long>(N_kv) * d_c > (1LL << 31))
        return fail(GBATTN_ERR_UNSUPPORTED, "mla_decode_host: problem too large");
    if (!Q_nope || !Q_pe || !KV_latent || !K_pe || !O || !LSE)
        return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_host: null tensor pointer");
    const size_t need = mla_decode_host_device_bytes(B, H, N_kv, d_c, d_r);
    if (!device_buf || device_bytes < need || (reinterpret_cast<uintptr_t>(device_buf) & 255u))
        return fail(GBATTN_ERR_WORKSPACE, "mla_decode_host: device buffer missing, smaller than "
                                          "mla_decode_host_device_bytes() or not 256-byte aligned");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    HostPipe *hp = nullptr;
    if ((rc = host_pipe(hp)) != GBATTN_OK) return rc;
    std::lock_guard<std::mutex> lk(hp->mu);

    const size_t qn_u = static_cast<size_t>(H) * d_c * 2, qp_u = static_cast<size_t>(H) * d_r * 2,
                 kv_u = static_cast<size_t>(N_kv) * d_c * 2, kp_u = static_cast<size_t>(N_kv) * d_r * 2,
                 o_u = static_cast<size_t>(H) * d_c * 2, l_u = static_cast<size_t>(H) * 4;
    uint8_t *dQn = static_cast<uint8_t *>(device_buf), *dQp = dQn + round256(B * qn_u),
            *dKV = dQp + round256(B * qp_u), *dKp = dKV + round256(B * kv_u), *dO = dKp + round256(B * kp_u),
            *dL = dO + round256(B * o_u), *dW = dL + round256(B * l_u);
    const size_t ws_bytes = mla_host_chunk_workspace(B, H, N_kv, d_c, env.num_sms);
    const int nchunk = std::min(kMlaChunks, B);
    cudaError_t e = pipe_start(hp, env.stream);
    std::string err;
    for (int c = 0; c < nchunk && e == cudaSuccess; ++c) {
        const int b0 = static_cast<int>(static_cast<long long>(c) * B / nchunk);
        const int b1 = static_cast<int>(static_cast<long long>(c + 1) * B / nchunk);
        const size_t nb = static_cast<size_t>(b1 - b0);
        const Piece in[4] = {{dQn + b0 * qn_u, static_cast<const uint8_t *>(Q_nope) + b0 * qn_u, nb * qn_u},
                             {dQp + b0 * qp_u, static_cast<const uint8_t *>(Q_pe) + b0 * qp_u, nb * qp_u},
                             {dKV + b0 * kv_u, static_cast<const uint8_t *>(KV_latent) + b0 * kv_u, nb * kv_u},
                             {dKp + b0 * kp_u, static_cast<const uint8_t *>(K_pe) + b0 * kp_u, nb * kp_u}};
        e = pipe_copy_in(hp, c, in, env.stream);
        if (e != cudaSuccess) break;
        // chunks run one after another on the caller's stream, so they share the workspace
        rc = launch_mla_decode(dQn + b0 * qn_u, dQp + b0 * qp_u, dKV + b0 * kv_u, dKp + b0 * kp_u, dO + b0 * o_u,
                               reinterpret_cast<float *>(dL + b0 * l_u), static_cast<int>(nb), H, N_kv, d_c, d_r,
                               scale, dW, ws_bytes, env, err);
        if (rc != GBATTN_OK) {
            g_err = err;
            return rc;
        }
        e = cudaEventRecord(hp->ev_k[c], env.stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->ev_k[c], 0);
        const Piece out[2] = {{static_cast<uint8_t *>(O) + b0 * o_u, dO + b0 * o_u, nb * o_u},
                              {reinterpret_cast<uint8_t *>(LSE) + b0 * l_u, dL + b0 * l_u, nb * l_u}};
        for (const Piece &pc : out)
            if (e == cudaSuccess) e = cudaMemcpyAsync(pc.dst, pc.src, pc.bytes, cudaMemcpyDeviceToHost, hp->d2h);
    }
    if (e == cudaSuccess) e = cudaEventRecord(hp->ev_out, hp->d2h);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(env.stream, hp->ev_out, 0);
    if (e != cudaSuccess) return fail(GBATTN_ERR_LAUNCH, std::string("mla_decode_host: ") + cudaGetErrorString(e));
    return GBATTN_OK;
}

extern "C" int gbattn_check(void *stream)
{
    g_err.clear();
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(env.stream);
    if (e != cudaSuccess) return fail(GBATTN_ERR_LAUNCH, std::string("stream: ") + cudaGetErrorString(e));
    int word = 0;
    e = cudaMemcpy(&word, env.status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(GBATTN_ERR_LAUNCH, std::string("status read: ") + cudaGetErrorString(e));
    if (word != 0) {
        cudaMemset(env.status, 0, sizeof(int));
        cudaDeviceSynchronize();
        if (word == kStatusBadLength)
            return fail(GBATTN_ERR_INVALID_ARG, "mla_decode_paged: a cache_seqlens entry was negative or "
                                                "beyond max_pages_per_seq * page_size (clamped; results invalid)");
        return fail(GBATTN_ERR_TIMEOUT, "a device-side bounded wait ran out; results of the "
                                        "affected launches are invalid");
    }
    return GBATTN_OK;
}

extern "C" const char *gbattn_last_error(void)
{
    return g_err.c_str();
}

extern "C" uint64_t gbattn_set_wait_timeout_ns(uint64_t ns)
{
    if (ns < 1000000ull) ns = 1000000ull;
    if (ns > 60000000000ull) ns = 60000000000ull;
    return g_timeout_ns.exchange(ns);
}

extern "C" int gbattn_set_fault_injection(int mode)
{
    if (mode < 0 || mode > 2) mode = 0;
    return g_inject.exchange(mode);
}

extern "C" int gbattn_mla_trace(void *host, size_t bytes)
{
    std::string err;
    const int rc = mla_trace_fetch(host, bytes, err);
    if (rc != GBATTN_OK) return fail(rc, err);
    return GBATTN_OK;
}

extern "C" int gbattn_attn_trace(void *host, size_t bytes)
{
    std::string err;
    const int rc = attn_trace_fetch(host, bytes, err);
    if (rc != GBATTN_OK) return fail(rc, err);
    return GBATTN_OK;
}

extern "C" int gbattn_selftest_umma(const void *A, const void *B, const void *P, const void *V, float *S,
                                    float *O, void *stream)
{
    g_err.clear();
    if (!A || !B || !P || !V || !S || !O) return fail(GBATTN_ERR_INVALID_ARG, "selftest: null pointer");
    if (!aligned16(A) || !aligned16(B) || !aligned16(P) || !aligned16(V) || !aligned16(S) || !aligned16(O))
        return fail(GBATTN_ERR_ALIGNMENT, "selftest: buffers must be 16-byte aligned");
    LaunchEnv env;
    int rc = get_env(env, stream);
    if (rc != GBATTN_OK) return rc;
    std::string err;
    rc = launch_selftest_umma(A, B, P, V, S, O, env, err);
    if (rc != GBATTN_OK) g_err = err;
    return rc;
}
