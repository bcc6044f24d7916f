// lm_head.cu -- projection of the verified rows to vocab logits.
//
// logits[n][v] = sum_h hid[n][h] W[h][v] (fp32 accumulation).  At k+1 rows
// per sequence the product is bound by streaming W once from HBM ([wmrh.cn
// tutorial, sec. 1.1]: every forward reads the weights once), so the kernel
// is built around the W stream:
//   * persistent CTAs walk 128-column slabs of W; each slab is K-looped in
//     64-row stages that TMA (cp.async.bulk.tensor, 128-byte swizzle) brings
//     into a multi-stage shared-memory ring, together with the matching
//     64-column slice of the hidden rows;
//   * the tensor cores take W^T as the M operand (ldmatrix.trans from the
//     swizzled tile) and the hidden rows as N (8..64 rows per pass), so the
//     vocab dimension fills the 16-row M side and tiny row counts waste no
//     MMA work;
//   * the epilogue transposes the fp32 tile through shared memory and writes
//     each logits row with coalesced 16-byte stores;
//   * optionally the epilogue also summarises each row of the slab by its
//     greedy argmax key (largest logit, lowest column; one 64-bit word per
//     row and slab), so greedy acceptance ([SpecDec-Context-Scaling guide,
//     sec. 3]) needs neither a second pass over the logits nor, when only
//     tokens are wanted, the logits at all.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kVT = 128;        // vocab columns per slab
constexpr int kHK = 64;         // hidden rows per stage
constexpr int kStages = 4;
constexpr int kThreads = 128;   // warp w owns columns [32w, 32w+32) of the slab
constexpr int kOutPitch = kVT + 4;

template <int NT>
struct LmSmem {
    static constexpr int NP = NT * 8;                      // rows per pass, padded
    static constexpr int kWBytes = kHK * kVT * 2;          // 16 KB: two 64x64 boxes
    static constexpr int kHBytes = NP * kHK * 2;           // NP x 64 box
    static constexpr int kStageBytes = kWBytes + kHBytes;  // multiple of 1024
    static constexpr int kOutBytes = NP * kOutPitch * 4;
    static constexpr int kTotal = kStages * kStageBytes + kOutBytes + kStages * 8 + 1024;
};

template <int NT>
__global__ void __launch_bounds__(kThreads) lm_head_kernel(const __grid_constant__ CUtensorMap tmW,
                                                          const __grid_constant__ CUtensorMap tmH,
                                                          float* __restrict__ logits, uint64_t* __restrict__ amax,
                                                          int N, int H, int V, int n0, int nslab, int w_ready,
                                                          unsigned int* err) {
    using S = LmSmem<NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* out_s = reinterpret_cast<float*>(smem + kStages * S::kStageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * S::kStageBytes + S::kOutBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nk = (H + kHK - 1) / kHK;
    const int my_slabs = blockIdx.x < nslab ? (nslab - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int total_it = my_slabs * nk;

    if (tid == 0) {
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmH);
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue_w = [&](int it) {   // W of step it (and the stage's whole byte count)
        const int slab = blockIdx.x + (it / nk) * gridDim.x;
        const int kc = it % nk;
        const int s = it % kStages;
        uint8_t* st = smem + s * S::kStageBytes;
        mbar_arrive_expect_tx(&full[s], S::kStageBytes);
        tma_load_2d(st, &tmW, slab * kVT, kc * kHK, &full[s]);
        tma_load_2d(st + kHK * 128, &tmW, slab * kVT + 64, kc * kHK, &full[s]);
    };
    auto issue_h = [&](int it) {   // the hidden rows' slice of step it
        const int kc = it % nk;
        const int s = it % kStages;
        tma_load_2d(smem + s * S::kStageBytes + S::kWBytes, &tmH, kc * kHK, n0, &full[s]);
    };
    auto issue = [&](int it) {
        issue_w(it);
        issue_h(it);
    };
    // The hidden rows come from the kernels before this one.  With w_ready the
    // weights are final before the preceding kernel runs, so the first ring
    // pass of W is on its way before waiting for it.
    const int npre = total_it < kStages ? total_it : kStages;
    if (w_ready && tid == 0)
        for (int it = 0; it < npre; ++it) issue_w(it);
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0)
        for (int it = 0; it < npre; ++it) {
            if (!w_ready) issue_w(it);
            issue_h(it);
        }

    float acc[2][NT][4];
    int it = 0;
    for (int si = 0; si < my_slabs; ++si) {
        const int slab = blockIdx.x + si * gridDim.x;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f;

        for (int kc = 0; kc < nk; ++kc, ++it) {
            const int s = it % kStages;
            mbar_wait(&full[s], (it / kStages) & 1, err);
            const uint32_t wbase = smem_u32(smem + s * S::kStageBytes) + (warp >> 1) * (kHK * 128);
            const uint32_t hbase = smem_u32(smem + s * S::kStageBytes + S::kWBytes);
#pragma unroll
            for (int ks = 0; ks < kHK / 16; ++ks) {
                uint32_t a[2][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    // W^T tile: v = (32*warp + 16*mt) % 64 + {0..15}, h = 16*ks + {0..15}
                    const int mi = lane >> 3, r = lane & 7;
                    const int hrow = ks * 16 + (mi >> 1) * 8 + r;
                    const int vcol = ((warp & 1) * 32 + mt * 16) + (mi & 1) * 8;
                    ldsm_x4_t(swz128(wbase, hrow, vcol >> 3), a[mt][0], a[mt][1], a[mt][2], a[mt][3]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    uint32_t b0, b1;
                    const int n = nt * 8 + (lane & 7);
                    const int chunk = ks * 2 + ((lane >> 3) & 1);
                    ldsm_x2(swz128(hbase, n, chunk), b0, b1);
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) mma_bf16(acc[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b0, b1);
                }
            }
            __syncthreads();   // stage s fully read
            if (tid == 0 && it + kStages < total_it) issue(it + kStages);
        }

        // epilogue: acc -> out_s[n][v] -> logits rows
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int v = warp * 32 + mt * 16 + (lane >> 2);
                const int n = nt * 8 + 2 * (lane & 3);
                out_s[n * kOutPitch + v] = acc[mt][nt][0];
                out_s[(n + 1) * kOutPitch + v] = acc[mt][nt][1];
                out_s[n * kOutPitch + v + 8] = acc[mt][nt][2];
                out_s[(n + 1) * kOutPitch + v + 8] = acc[mt][nt][3];
            }
        __syncthreads();
        const int vbase = slab * kVT;
        const int nrows = min(S::NP, N - n0);
        if (amax) {
            // argmax key of each row over the slab: warp w takes rows w, w+4,
            // ...; lane l holds columns 4l..4l+3 (V % 4 == 0: all or none valid)
            bool nan_seen = false;
            for (int n = warp; n < nrows; n += kThreads / 32) {
                const int c = 4 * lane;
                uint64_t best = 0;
                if (vbase + c < V) {
                    const float4 x = *reinterpret_cast<const float4*>(out_s + n * kOutPitch + c);
                    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        nan_seen |= xs[e] != xs[e];
                        const uint64_t k = argmax_key(argmax_okey(xs[e]), vbase + c + e);
                        best = k > best ? k : best;
                    }
                }
                best = warp_max_key(best);
                if (lane == 0) amax[static_cast<size_t>(n0 + n) * nslab + slab] = best;
            }
            if (__any_sync(0xffffffffu, nan_seen) && lane == 0) raise_error(err, SV_DEVERR_NONFINITE);
        }
        if (logits)
            for (int x = tid; x < nrows * (kVT / 4); x += kThreads) {
                const int n = x / (kVT / 4), c = (x % (kVT / 4)) * 4;
                if (vbase + c < V) {
                    const float4 val = *reinterpret_cast<const float4*>(out_s + n * kOutPitch + c);
                    *reinterpret_cast<float4*>(logits + static_cast<size_t>(n0 + n) * V + vbase + c) = val;
                }
            }
        __syncthreads();
    }
}

template <int NT>
cudaError_t launch_nt(const uint16_t* hid, const uint16_t* W, float* logits, uint64_t* amax, int N, int H, int V,
                      int n0, bool w_ready, cudaStream_t st) {
    using S = LmSmem<NT>;
    alignas(64) uint8_t tmW[128], tmH[128];
    if (!encode_tmap_2d_bf16(tmW, W, V, H, static_cast<uint64_t>(V) * 2, 64, kHK)) return cudaErrorInvalidValue;
    if (!encode_tmap_2d_bf16(tmH, hid, H, N, static_cast<uint64_t>(H) * 2, kHK, S::NP)) return cudaErrorInvalidValue;
    static PerDeviceOnce attr_once;
    const cudaError_t ea = attr_once.run([]() {
        return cudaFuncSetAttribute(lm_head_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
    });
    if (ea != cudaSuccess) return ea;
    const int nslab = (V + kVT - 1) / kVT;
    const int per_sm = S::kTotal <= 110 * 1024 ? 2 : 1;
    int grid = device_sm_count() * per_sm;
    if (grid > nslab) grid = nslab;
    return launch_pdl(lm_head_kernel<NT>, dim3(grid), dim3(kThreads), S::kTotal, st,
                      *reinterpret_cast<const CUtensorMap*>(tmW), *reinterpret_cast<const CUtensorMap*>(tmH), logits, amax,
                      N, H, V, n0, nslab, w_ready ? 1 : 0, device_error_word());
}

}  // namespace

cudaError_t launch_lm_head(const uint16_t* hid, const uint16_t* W, float* logits, uint64_t* amax, int N, int H,
                           int V, bool w_ready, cudaStream_t st) {
    // Beyond 16 rows the product is a real dense contraction: tcgen05, up to
    // 256 rows per pass over W.
    if (N > 16) {
        for (int n0 = 0; n0 < N; n0 += 256) {
            const int rows = N - n0 < 256 ? N - n0 : 256;
            const cudaError_t e = launch_lm_head_tc(hid, W, logits, amax, N, H, V, n0, rows, w_ready, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    for (int n0 = 0; n0 < N; n0 += 64) {
        const int rows = N - n0 < 64 ? N - n0 : 64;
        const int nt = (rows + 7) / 8;
        cudaError_t e;
        switch (nt) {
            case 1: e = launch_nt<1>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
            case 2: e = launch_nt<2>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
            case 3: e = launch_nt<3>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
            case 4: e = launch_nt<4>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
            case 5: e = launch_nt<5>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
            case 6: e = launch_nt<6>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
            case 7: e = launch_nt<7>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
            default: e = launch_nt<8>(hid, W, logits, amax, N, H, V, n0, w_ready, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sv
