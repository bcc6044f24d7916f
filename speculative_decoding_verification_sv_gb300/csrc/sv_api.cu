// sv_api.cu -- extern "C" entry points of libsv.so (declared in include/sv.h).
//
// Each entry point validates what the host can see, then enqueues the
// kernels of its translation unit on the caller's stream.  The library
// allocates nothing: scratch comes from the caller's workspace, and the only
// library-owned device state is the error word below.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "sv.h"
#include "sv_internal.h"

namespace sv {

// Device error word: sticky bits raised by kernels (see SV_DEVERR_*),
// read and cleared by sv_get_device_error.
__device__ unsigned int g_error_word;

namespace {
std::mutex g_mu;
PerDeviceOnce g_err_once;
unsigned int* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
bool g_ctx_fns_looked_up = false;

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return (d >= 0 && d < kMaxDevices) ? d : 0;
}

template <typename P>
P driver_fn(const char* name, int version) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return reinterpret_cast<P>(fn);
}
}  // namespace

unsigned long long current_context_id() {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_ctx_fns_looked_up) {
            g_ctx_current = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
            g_ctx_id = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
            g_ctx_fns_looked_up = true;
        }
    }
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

unsigned int* device_error_word() {
    const int d = current_device();
    const cudaError_t e = g_err_once.run([d]() {
        void* p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_error_word);
        g_err_ptr[d] = r == cudaSuccess ? static_cast<unsigned int*>(p) : nullptr;
        return r;
    });
    if (e != cudaSuccess) return nullptr;
    return g_err_ptr[d];
}

int device_sm_count() {
    const int d = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = kSmCount;
        g_sm_count[d] = n;
    }
    return g_sm_count[d];
}

bool encode_tmap_2d_bf16(void* tmap, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                         uint32_t box_inner, uint32_t box_outer) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return false;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace sv

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline sv_status launch_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

int sv_version(void) { return 100; }

const char* sv_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "ok";
        case SV_ERR_ARG: return "invalid argument";
        case SV_ERR_SHAPE: return "invalid shape";
        case SV_ERR_UNSUPPORTED: return "unsupported configuration";
        case SV_ERR_WORKSPACE: return "workspace too small";
        case SV_ERR_CUDA: return "CUDA runtime error";
        case SV_ERR_DEVICE: return "device-side error bit set";
    }
    return "unknown status";
}

sv_status sv_get_device_error(uint32_t* word, void* stream) {
    unsigned int* p = sv::device_error_word();
    if (!p) return SV_ERR_CUDA;
    cudaStream_t st = as_stream(stream);
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, p, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, sizeof(unsigned int), st) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SV_ERR_CUDA;
    if (word) *word = host;
    return host ? SV_ERR_DEVICE : SV_OK;
}

// ---------------------------------------------------------------------------

static sv_status check_attn_shape(const sv_attn_shape* s) {
    if (!s) return SV_ERR_ARG;
    if (s->B < 1 || s->R < 1 || s->R > 128 || s->Hq < 1 || s->Hkv < 1 || s->T_cap < 1) return SV_ERR_SHAPE;
    if (s->Hq % s->Hkv != 0 || s->Hq / s->Hkv > 16) return SV_ERR_SHAPE;
    if (s->D != 128) return SV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(s->B) * s->Hkv * s->T_cap >= (int64_t(1) << 31)) return SV_ERR_SHAPE;
    if (static_cast<int64_t>(s->B) * s->Hkv > 65535) return SV_ERR_SHAPE;
    return SV_OK;
}

size_t sv_verify_attn_workspace(const sv_attn_shape* shape) {
    if (check_attn_shape(shape) != SV_OK) return 0;
    return sv::attn_workspace(*shape);
}

sv_status sv_verify_attn(const sv_attn_shape* shape, const uint16_t* q, const uint16_t* k_cache,
                         const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk, const uint16_t* v_blk,
                         const int32_t* parent, float scale, uint16_t* out, void* ws, size_t ws_bytes,
                         void* stream) {
    return sv_verify_attn_ex(shape, q, k_cache, v_cache, len, k_blk, v_blk, parent, scale, out, ws, ws_bytes, 0u,
                             stream);
}

sv_status sv_verify_attn_ex(const sv_attn_shape* shape, const uint16_t* q, const uint16_t* k_cache,
                            const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk,
                            const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out, void* ws,
                            size_t ws_bytes, uint32_t flags, void* stream) {
    if (flags & ~SV_ATTN_CACHE_READY) return SV_ERR_ARG;
    const sv_status st = check_attn_shape(shape);
    if (st != SV_OK) return st;
    if (!q || !k_cache || !v_cache || !len || !k_blk || !v_blk || !out) return SV_ERR_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_blk) || !aligned16(v_blk) ||
        !aligned16(out) || (ws && !aligned16(ws)))
        return SV_ERR_ARG;
    if (!ws && sv::attn_workspace(*shape) > 0) return SV_ERR_ARG;
    if (!(scale > 0.0f)) return SV_ERR_ARG;
    if (ws_bytes < sv::attn_workspace(*shape)) return SV_ERR_WORKSPACE;
    return launch_status(sv::launch_verify_attn(*shape, q, k_cache, v_cache, len, k_blk, v_blk, parent, scale, out,
                                                ws, (flags & SV_ATTN_CACHE_READY) != 0, nullptr, 0, 0,
                                                as_stream(stream)));
}

sv_status sv_verify_attn_paged(const sv_attn_shape* shape, const uint16_t* q, const uint16_t* k_pool,
                               const uint16_t* v_pool, int32_t num_pages, const int32_t* page_table,
                               int32_t max_pages, const int32_t* len, const uint16_t* k_blk, const uint16_t* v_blk,
                               const int32_t* parent, float scale, uint16_t* out, void* ws, size_t ws_bytes,
                               uint32_t flags, void* stream) {
    if (flags & ~SV_ATTN_CACHE_READY) return SV_ERR_ARG;
    const sv_status st = check_attn_shape(shape);
    if (st != SV_OK) return st;
    if (!q || !k_pool || !v_pool || !page_table || !len || !k_blk || !v_blk || !out) return SV_ERR_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_blk) || !aligned16(v_blk) ||
        !aligned16(out) || (ws && !aligned16(ws)))
        return SV_ERR_ARG;
    if (num_pages < 1 || max_pages < 1) return SV_ERR_SHAPE;
    if (static_cast<int64_t>(max_pages) * SV_KV_PAGE != shape->T_cap) return SV_ERR_SHAPE;
    // tensor-map rows of the pool, and the out-of-pool row used for a bad entry
    if ((static_cast<int64_t>(num_pages) + 1) * shape->Hkv * SV_KV_PAGE >= (int64_t(1) << 31)) return SV_ERR_SHAPE;
    if (!ws && sv::attn_workspace(*shape) > 0) return SV_ERR_ARG;
    if (!(scale > 0.0f)) return SV_ERR_ARG;
    if (ws_bytes < sv::attn_workspace(*shape)) return SV_ERR_WORKSPACE;
    return launch_status(sv::launch_verify_attn(*shape, q, k_pool, v_pool, len, k_blk, v_blk, parent, scale, out, ws,
                                                (flags & SV_ATTN_CACHE_READY) != 0, page_table, max_pages,
                                                num_pages, as_stream(stream)));
}

sv_status sv_lm_head(const uint16_t* hid, const uint16_t* W, float* logits, int32_t N, int32_t H, int32_t V,
                     void* stream) {
    return sv_lm_head_ex(hid, W, logits, N, H, V, 0u, stream);
}

sv_status sv_lm_head_ex(const uint16_t* hid, const uint16_t* W, float* logits, int32_t N, int32_t H, int32_t V,
                        uint32_t flags, void* stream) {
    if (flags & ~SV_LM_WEIGHTS_READY) return SV_ERR_ARG;
    if (!hid || !W || !logits) return SV_ERR_ARG;
    if (!aligned16(hid) || !aligned16(W) || !aligned16(logits)) return SV_ERR_ARG;
    if (N < 1 || N > 4096 || H < 8 || V < 8 || H % 8 || V % 8) return SV_ERR_SHAPE;
    return launch_status(sv::launch_lm_head(hid, W, logits, nullptr, N, H, V, (flags & SV_LM_WEIGHTS_READY) != 0,
                                            as_stream(stream)));
}

size_t sv_lm_head_argmax_bytes(int32_t N, int32_t V) {
    if (N < 1 || V < 1) return 0;
    return static_cast<size_t>(N) * ((V + SV_ARGMAX_SLAB - 1) / SV_ARGMAX_SLAB) * sizeof(uint64_t);
}

sv_status sv_lm_head_argmax(const uint16_t* hid, const uint16_t* W, float* logits, int32_t N, int32_t H, int32_t V,
                            uint64_t* argmax, size_t argmax_bytes, uint32_t flags, void* stream) {
    if (flags & ~SV_LM_WEIGHTS_READY) return SV_ERR_ARG;
    if (!hid || !W || !argmax) return SV_ERR_ARG;
    if (!aligned16(hid) || !aligned16(W) || !aligned16(argmax) || (logits && !aligned16(logits))) return SV_ERR_ARG;
    if (N < 1 || N > 4096 || H < 8 || V < 8 || H % 8 || V % 8) return SV_ERR_SHAPE;
    if (argmax_bytes < sv_lm_head_argmax_bytes(N, V)) return SV_ERR_WORKSPACE;
    return launch_status(sv::launch_lm_head(hid, W, logits, argmax, N, H, V, (flags & SV_LM_WEIGHTS_READY) != 0,
                                            as_stream(stream)));
}

sv_status sv_accept_greedy_commit(const uint64_t* argmax, const int32_t* tok, const int32_t* parent, int32_t B,
                                  int32_t R, int32_t V, int32_t* n_acc, int32_t* out_tok, int32_t* path,
                                  uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk,
                                  int32_t L, int32_t Hkv, int32_t D, int32_t T_cap, int32_t* len, void* stream) {
    if (!argmax || !tok || !n_acc || !out_tok || !path) return SV_ERR_ARG;
    if (!aligned16(argmax)) return SV_ERR_ARG;
    if (B < 1 || R < 1 || R > 128 || V < 1 || static_cast<int64_t>(B) * 8 > 2147483647) return SV_ERR_SHAPE;
    const bool commit = k_cache != nullptr;
    if (commit) {
        if (!v_cache || !k_blk || !v_blk || !len) return SV_ERR_ARG;
        if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_blk) || !aligned16(v_blk)) return SV_ERR_ARG;
        if (L < 1 || Hkv < 1 || D < 8 || D % 8 || T_cap < 1) return SV_ERR_SHAPE;
    } else if (v_cache || k_blk || v_blk) {
        return SV_ERR_ARG;   // a commit needs all four buffers
    }
    return launch_status(sv::launch_accept_greedy_commit(argmax, tok, parent, B, R, V, n_acc, out_tok, path,
                                                         commit ? k_cache : nullptr, v_cache, k_blk, v_blk, L, Hkv, D,
                                                         T_cap, len, nullptr, 0, 0, as_stream(stream)));
}

sv_status sv_accept_greedy_commit_paged(const uint64_t* argmax, const int32_t* tok, const int32_t* parent, int32_t B,
                                        int32_t R, int32_t V, int32_t* n_acc, int32_t* out_tok, int32_t* path,
                                        uint16_t* k_pool, uint16_t* v_pool, int32_t num_pages,
                                        const int32_t* page_table, int32_t max_pages, const uint16_t* k_blk,
                                        const uint16_t* v_blk, int32_t L, int32_t Hkv, int32_t D, int32_t* len,
                                        void* stream) {
    if (!argmax || !tok || !n_acc || !out_tok || !path) return SV_ERR_ARG;
    if (!k_pool || !v_pool || !page_table || !k_blk || !v_blk || !len) return SV_ERR_ARG;
    if (!aligned16(argmax) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_blk) || !aligned16(v_blk))
        return SV_ERR_ARG;
    if (B < 1 || R < 1 || R > 128 || V < 1 || static_cast<int64_t>(B) * 8 > 2147483647) return SV_ERR_SHAPE;
    if (L < 1 || Hkv < 1 || D < 8 || D % 8 || num_pages < 1 || max_pages < 1) return SV_ERR_SHAPE;
    if (static_cast<int64_t>(max_pages) * SV_KV_PAGE > 2147483647) return SV_ERR_SHAPE;
    return launch_status(sv::launch_accept_greedy_commit(argmax, tok, parent, B, R, V, n_acc, out_tok, path, k_pool,
                                                         v_pool, k_blk, v_blk, L, Hkv, D, max_pages * SV_KV_PAGE, len,
                                                         page_table, max_pages, num_pages, as_stream(stream)));
}

size_t sv_accept_greedy_workspace(int32_t B, int32_t R, int32_t V) {
    if (B < 1 || R < 1 || V < 1) return 0;
    return sv::greedy_workspace(B, R, V);
}

sv_status sv_accept_greedy(const float* logits, const int32_t* tok, const int32_t* parent, int32_t B, int32_t R,
                           int32_t V, int32_t* n_acc, int32_t* out_tok, int32_t* path, void* ws, size_t ws_bytes,
                           void* stream) {
    if (!logits || !tok || !n_acc || !out_tok || !path || !ws) return SV_ERR_ARG;
    if (!aligned16(logits) || !aligned16(ws)) return SV_ERR_ARG;
    if (B < 1 || R < 1 || R > 128 || V < 1 || static_cast<int64_t>(B) * R > 65535) return SV_ERR_SHAPE;
    if (ws_bytes < sv::greedy_workspace(B, R, V)) return SV_ERR_WORKSPACE;
    return launch_status(
        sv::launch_accept_greedy(logits, tok, parent, B, R, V, n_acc, out_tok, path, ws, as_stream(stream)));
}

size_t sv_accept_greedy_relaxed_workspace(int32_t B, int32_t R, int32_t V) {
    if (B < 1 || R < 1 || V < 1) return 0;
    return sv::relaxed_workspace(B, R, V);
}

sv_status sv_accept_greedy_relaxed(const float* logits, const int32_t* tok, const int32_t* parent, int32_t B,
                                   int32_t R, int32_t V, float delta, int32_t* n_acc, int32_t* out_tok,
                                   int32_t* path, void* ws, size_t ws_bytes, void* stream) {
    if (!logits || !tok || !n_acc || !out_tok || !path || !ws) return SV_ERR_ARG;
    if (!(delta >= 0.0f)) return SV_ERR_ARG;   // negative or NaN
    if (!aligned16(ws)) return SV_ERR_ARG;
    if (B < 1 || R < 1 || R > 128 || V < 1 || static_cast<int64_t>(B) * R > 65535) return SV_ERR_SHAPE;
    if (ws_bytes < sv::relaxed_workspace(B, R, V)) return SV_ERR_WORKSPACE;
    return launch_status(sv::launch_accept_relaxed(logits, tok, parent, B, R, V, delta, n_acc, out_tok, path, ws,
                                                   as_stream(stream)));
}

size_t sv_accept_sample_workspace(int32_t B, int32_t R, int32_t V) {
    if (B < 1 || R < 1 || V < 1) return 0;
    return sv::sample_workspace(B, R, V);
}

sv_status sv_accept_sample(const float* logits, const float* q, int32_t Vq, const int32_t* tok,
                           const int32_t* parent, int32_t B, int32_t R, int32_t V, float temperature, uint64_t seed,
                           uint64_t step, const float* uniforms, int32_t* n_acc, int32_t* out_tok, int32_t* path,
                           void* ws, size_t ws_bytes, void* stream) {
    if (!logits || !tok || !n_acc || !out_tok || !path || !ws) return SV_ERR_ARG;
    if (R > 1 || parent) {
        if (!q) return SV_ERR_ARG;
        if (!aligned16(q)) return SV_ERR_ARG;
    }
    if (!aligned16(logits) || !aligned16(ws)) return SV_ERR_ARG;
    if (!(temperature > 0.0f) || !(temperature < 1e30f)) return SV_ERR_ARG;
    if (B < 1 || R < 1 || R > 128 || V < 4 || V > (1 << 18) || V % 4) return SV_ERR_SHAPE;
    if (Vq < 4 || Vq > V || Vq % 4) return SV_ERR_SHAPE;
    if (static_cast<int64_t>(B) * R * 8 > (int64_t(1) << 31) - 1) return SV_ERR_SHAPE;
    if (ws_bytes < sv::sample_workspace(B, R, V)) return SV_ERR_WORKSPACE;
    return launch_status(sv::launch_accept_sample(logits, q, Vq, tok, parent, B, R, V, temperature, seed, step,
                                                  uniforms, n_acc, out_tok, path, ws, ws_bytes, as_stream(stream)));
}

sv_status sv_kv_commit(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk, int32_t L,
                       int32_t B, int32_t Hkv, int32_t D, int32_t T_cap, int32_t R, const int32_t* path,
                       const int32_t* n_acc, int32_t* len, void* stream) {
    if (!k_cache || !v_cache || !k_blk || !v_blk || !path || !n_acc || !len) return SV_ERR_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_blk) || !aligned16(v_blk)) return SV_ERR_ARG;
    if (L < 1 || B < 1 || Hkv < 1 || D < 8 || D % 8 || T_cap < 1 || R < 1 || R > 128) return SV_ERR_SHAPE;
    if (static_cast<int64_t>(B) * 8 > 2147483647) return SV_ERR_SHAPE;
    return launch_status(sv::launch_kv_commit(k_cache, v_cache, k_blk, v_blk, L, B, Hkv, D, T_cap, R, path, n_acc, len,
                                              nullptr, 0, 0, as_stream(stream)));
}

sv_status sv_kv_commit_paged(uint16_t* k_pool, uint16_t* v_pool, int32_t num_pages, const int32_t* page_table,
                             int32_t max_pages, const uint16_t* k_blk, const uint16_t* v_blk, int32_t L, int32_t B,
                             int32_t Hkv, int32_t D, int32_t R, const int32_t* path, const int32_t* n_acc, int32_t* len,
                             void* stream) {
    if (!k_pool || !v_pool || !page_table || !k_blk || !v_blk || !path || !n_acc || !len) return SV_ERR_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_blk) || !aligned16(v_blk)) return SV_ERR_ARG;
    if (L < 1 || B < 1 || Hkv < 1 || D < 8 || D % 8 || R < 1 || R > 128 || num_pages < 1 || max_pages < 1)
        return SV_ERR_SHAPE;
    if (static_cast<int64_t>(max_pages) * SV_KV_PAGE > 2147483647 || static_cast<int64_t>(B) * 8 > 2147483647)
        return SV_ERR_SHAPE;
    return launch_status(sv::launch_kv_commit(k_pool, v_pool, k_blk, v_blk, L, B, Hkv, D, max_pages * SV_KV_PAGE, R,
                                              path, n_acc, len, page_table, max_pages, num_pages,
                                              as_stream(stream)));
}

// Device or page-locked host memory (the kernel reaches both through unified
// addressing); pageable or unknown pointers are refused.
static bool gpu_reachable(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

sv_status sv_copy(void* dst, const void* src, size_t bytes, void* stream) {
    if (bytes == 0) return SV_OK;
    if (!dst || !src) return SV_ERR_ARG;
    if (!gpu_reachable(dst) || !gpu_reachable(src)) return SV_ERR_ARG;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (d < s + bytes && s < d + bytes) return SV_ERR_ARG;   // overlapping ranges
    return launch_status(sv::launch_stage_copy(dst, src, bytes, as_stream(stream)));
}

sv_status sv_diag_exp(const float* x, float* y, int64_t n, void* stream) {
    if (n < 0 || (n > 0 && (!x || !y))) return SV_ERR_ARG;
    if (n == 0) return SV_OK;
    return launch_status(sv::launch_diag_exp(x, y, n, as_stream(stream)));
}

sv_status sv_diag_div(const float* a, const float* b, float* q, int64_t n, void* stream) {
    if (n < 0 || (n > 0 && (!a || !b || !q))) return SV_ERR_ARG;
    if (n == 0) return SV_OK;
    return launch_status(sv::launch_diag_div(a, b, q, n, as_stream(stream)));
}

sv_status sv_diag_philox(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int64_t n, void* stream) {
    if (n < 0 || (n > 0 && (!ctr || !key || !out))) return SV_ERR_ARG;
    if (n == 0) return SV_OK;
    return launch_status(sv::launch_diag_philox(ctr, key, out, n, as_stream(stream)));
}

sv_status sv_diag_canon(const float* x, int32_t n, int32_t m, const float* u, float* sums, int32_t* draws,
                        void* stream) {
    if (!x || !u || !sums || !draws) return SV_ERR_ARG;
    if (!aligned16(x)) return SV_ERR_ARG;
    if (n < 4 || n > (1 << 18) || n % 4 || m < 1 || m > 65535) return SV_ERR_SHAPE;
    return launch_status(sv::launch_diag_canon(x, n, m, u, sums, draws, as_stream(stream)));
}

}  // extern "C"
