// sv_internal.h -- launchers shared between the kernel translation units and
// the C-ABI entry points (sv_api.cu).  Host-side only; not installed.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "sv.h"

namespace sv {

constexpr int kMaxDevices = 64;

// Identity of the calling thread's current CUDA context (cuCtxGetId); 0 when
// no context is current or the query is unavailable.  A device reset
// (cudaDeviceReset) ends the context, and the next one gets another id, so
// set-up keyed on it is redone on the new context.
unsigned long long current_context_id();

// One-time set-up per device and context (kernel attributes, symbol
// addresses): run() calls `f` on the current device the first time it is
// asked there, and again after that device's context has been replaced.
// Thread-safe; `f` runs under the object's lock.
class PerDeviceOnce {
public:
    template <typename F>
    cudaError_t run(F&& f) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lk(mu_);
        const unsigned long long before = current_context_id();
        if (done_[dev] && before == ctx_[dev]) return cudaSuccess;
        const cudaError_t e = f();
        if (e != cudaSuccess) return e;
        done_[dev] = true;
        ctx_[dev] = current_context_id();   // f made the context current if it was not
        return cudaSuccess;
    }

private:
    std::mutex mu_;
    bool done_[kMaxDevices] = {};
    unsigned long long ctx_[kMaxDevices] = {};
};

// Launch with programmatic dependent launch allowed: the kernel may start
// while the previous kernel on the stream drains, and waits
// (griddepcontrol.wait) before it touches anything that kernel produced.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

constexpr int kSmCount = 152;   // GB300; launch heuristics query the device when it differs

unsigned int* device_error_word();          // per-device __device__ word (sv_api.cu)
int device_sm_count();

// accept.cu
size_t greedy_workspace(int B, int R, int V);
cudaError_t launch_accept_greedy(const float* logits, const int32_t* tok, const int32_t* parent, int B, int R,
                                 int V, int32_t* n_acc, int32_t* out_tok, int32_t* path, void* ws,
                                 cudaStream_t st);
// accept_relaxed.cu
size_t relaxed_workspace(int B, int R, int V);
cudaError_t launch_accept_relaxed(const float* logits, const int32_t* tok, const int32_t* parent, int B, int R, int V,
                                  float delta, int32_t* n_acc, int32_t* out_tok, int32_t* path, void* ws,
                                  cudaStream_t st);
// accept.cu (sampled)
size_t sample_workspace(int B, int R, int V);
cudaError_t launch_accept_sample(const float* logits, const float* q, int Vq, const int32_t* tok,
                                 const int32_t* parent, int B, int R, int V, float temperature, uint64_t seed,
                                 uint64_t step, const float* uniforms, int32_t* n_acc, int32_t* out_tok,
                                 int32_t* path, void* ws, size_t ws_bytes, cudaStream_t st);
// stage.cu
cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, cudaStream_t st);
cudaError_t launch_diag_exp(const float* x, float* y, int64_t n, cudaStream_t st);
cudaError_t launch_diag_div(const float* a, const float* b, float* q, int64_t n, cudaStream_t st);
cudaError_t launch_diag_philox(const uint32_t* ctr, const uint32_t* key, uint32_t* out, int64_t n,
                               cudaStream_t st);
cudaError_t launch_diag_canon(const float* x, int n, int m, const float* u, float* sums, int32_t* draws,
                              cudaStream_t st);

// kv_commit.cu
// pages != nullptr: the caches are page pools [L][num_pages][Hkv][64][D] and
// pages [B][max_pages] maps each 64-position tile to its page (T_cap =
// max_pages * 64)
cudaError_t launch_kv_commit(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk,
                             int L, int B, int Hkv, int D, int T_cap, int R, const int32_t* path,
                             const int32_t* n_acc, int32_t* len, const int32_t* pages, int max_pages,
                             int num_pages, cudaStream_t st);

// kv_commit.cu: greedy acceptance from the LM head's argmax keys [B*R][nslab],
// then (k_cache != nullptr) the commit, in one launch; pages != nullptr: the
// caches are page pools as for launch_kv_commit
cudaError_t launch_accept_greedy_commit(const uint64_t* amax, const int32_t* tok, const int32_t* parent, int B, int R,
                                        int V, int32_t* n_acc, int32_t* out_tok, int32_t* path, uint16_t* k_cache,
                                        uint16_t* v_cache, const uint16_t* k_blk, const uint16_t* v_blk, int L,
                                        int Hkv, int D, int T_cap, int32_t* len, const int32_t* pages, int max_pages,
                                        int num_pages, cudaStream_t st);

// lm_head.cu.  logits may be nullptr (not written); amax nullptr or
// [N][ceil(V/128)] greedy argmax keys, one per row and 128-column slab.
constexpr int kArgmaxSlab = 128;
cudaError_t launch_lm_head(const uint16_t* hid, const uint16_t* W, float* logits, uint64_t* amax, int N, int H,
                           int V, bool w_ready, cudaStream_t st);

// lm_head_tc.cu (rows n0 .. n0+rows-1, 1 <= rows <= 256)
cudaError_t launch_lm_head_tc(const uint16_t* hid, const uint16_t* W, float* logits, uint64_t* amax, int N, int H,
                              int V, int n0, int rows, bool w_ready, cudaStream_t st);

// verify_attn.cu
struct AttnPlan {
    int G;          // query heads per KV head
    int rows;       // R * G query rows per (sequence, KV head)
    int row_tiles;  // ceil(rows / rows per tile)
    bool half;      // 64-row tiles (M = 64 MMAs), else 128-row tiles (M = 128); two key tiles per step in both
    bool hw4;       // half tiles with four row-owner warps per TMEM quadrant (long loops), else two
    bool split_kv;  // K and V halves of a ring stage on separate barriers (full tiles; half tiles whose loops
                    // are longer than the ring over one row tile)
    int warps;      // warps per CTA
    int splits;     // CTAs per thread-block cluster (split-KV merged through DSMEM)
    int clusters;   // clusters per (sequence, KV head, row tile); > 1 merges in the workspace
    bool xch;       // the cluster's CTAs exchange their partial rows through L2 (the workspace's
                    // exchange area) instead of pushing them into the owners' shared memory
};
AttnPlan attn_plan(const sv_attn_shape& s);
size_t attn_workspace(const sv_attn_shape& s);
// pages != nullptr: k_cache / v_cache are page pools [num_pages][Hkv][64][D]
// and pages [B][max_pages] maps each 64-position tile to its page
cudaError_t launch_verify_attn(const sv_attn_shape& s, const uint16_t* q, const uint16_t* k_cache,
                               const uint16_t* v_cache, const int32_t* len, const uint16_t* k_blk,
                               const uint16_t* v_blk, const int32_t* parent, float scale, uint16_t* out,
                               void* ws, bool cache_ready, const int32_t* pages, int max_pages, int num_pages,
                               cudaStream_t st);

// TMA descriptor encoding (driver entry point fetched through the runtime).
bool encode_tmap_2d_bf16(void* tmap, const void* base, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                         uint32_t box_inner, uint32_t box_outer);

}  // namespace sv
