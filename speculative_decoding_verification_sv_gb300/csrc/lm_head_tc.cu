// lm_head_tc.cu -- LM head on the 5th-generation tensor cores (tcgen05) for
// 17..256 verified rows per pass (many sequences, or a draft tree).
//
// logits[n][v] = sum_h hid[n][h] W[h][v].  With tens of rows the product is a
// real dense contraction (144 rows x 3584 x 152064 = 157 GFLOP against 1.1 GB
// of weights), so the tile is computed as D[v][n] = W^T[v][h] hid^T[h][n]:
//   * M = 128 vocab columns (A = W^T, read MN-major straight from the W tile
//     TMA brings in), N = all rows of the pass (B = hidden rows, K-major),
//     K = H in 64-wide stages;
//   * warp 4 issues the TMA copies into a ring of stages (full/empty mbarriers);
//   * one thread of warp 5 issues tcgen05.mma (4 per stage) into a TMEM
//     accumulator and releases each stage with tcgen05.commit;
//   * warps 0..3 read the accumulator (tcgen05.ld, one vocab column per
//     thread) and store each logits row with 128-byte coalesced writes;
//   * two TMEM accumulators alternate so a slab's epilogue overlaps the next
//     slab's MMAs; CTAs are persistent over 128-column slabs;
//   * optionally the epilogue also writes each row's greedy argmax key over
//     the slab (two redux steps per row and warp, then the four warps' keys
//     combined through shared memory), the summary greedy acceptance reads
//     in place of the logits.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kM = 128;          // vocab columns per slab (MMA M)
constexpr int kHK = 64;          // hidden rows per stage
constexpr int kThreads = 192;    // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int kWBytes = kHK * kM * 2;   // 16 KB: two 64x64 boxes

template <int NP>
struct TcCfg {
    static constexpr int kHBytes = NP * kHK * 2;
    static constexpr int kStageBytes = kWBytes + kHBytes;
    static constexpr int kArgBytes = 4 * NP * 8;   // argmax keys: [epilogue warp][row]
    // six stages where they fit beside the barriers and the argmax keys
    static constexpr int kStages = (kStageBytes * 6 + 1024 + 256 + kArgBytes <= 232448) ? 6 : 4;
    static constexpr int kAccCols = NP <= 32 ? 32 : NP <= 64 ? 64 : NP <= 128 ? 128 : 256;
    static constexpr int kTmemCols = 2 * kAccCols;
    static constexpr int kSmem = kStages * kStageBytes + 1024 + 256 + kArgBytes;
};

template <int NP>
__global__ void __launch_bounds__(kThreads, 1) lm_head_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                const __grid_constant__ CUtensorMap tmH,
                                                                float* __restrict__ logits,
                                                                uint64_t* __restrict__ amax, int N, int H, int V,
                                                                int n0, int nslab, int w_ready, unsigned int* err) {
    using C = TcCfg<NP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
    uint64_t* empty = full + C::kStages;
    uint64_t* acc_full = empty + C::kStages;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(acc_empty + 2);
    uint64_t* keys_s = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes + 256);   // [4][NP]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = (H + kHK - 1) / kHK;
    const int my_slabs = blockIdx.x < nslab ? (nslab - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmH);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 4);
        }
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(tmem_base_s, C::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_s;
    // The hidden rows come from the kernels before this one.  With w_ready the
    // weights are final before the preceding kernel runs: the producer issues
    // the first ring pass of W before waiting for it.
    const bool early = w_ready != 0;
    if (!early || warp != 4) {
        pdl_wait();
        pdl_launch_dependents();
    }

    if (warp == 4) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const int total_it = my_slabs * nk;
            // step it = slab si, hidden-row block kc (counters, no division per step)
            auto load_w = [&](int it, int si, int kc) {   // W of step it (and the stage's whole byte count)
                const int slab = blockIdx.x + si * gridDim.x, s = it % C::kStages;
                mbar_wait(&empty[s], ((it / C::kStages) & 1) ^ 1, err);
                uint8_t* st = smem + s * C::kStageBytes;
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                tma_load_2d(st, &tmW, slab * kM, kc * kHK, &full[s]);
                tma_load_2d(st + kHK * 128, &tmW, slab * kM + 64, kc * kHK, &full[s]);
            };
            auto load_h = [&](int it, int kc) {   // the hidden rows' slice of step it
                const int s = it % C::kStages;
                tma_load_2d(smem + s * C::kStageBytes + kWBytes, &tmH, kc * kHK, n0, &full[s]);
            };
            const int npre = early ? (total_it < C::kStages ? total_it : C::kStages) : 0;
            for (int it = 0, si = 0, kc = 0; it < npre; ++it) {
                load_w(it, si, kc);
                if (++kc == nk) { kc = 0; ++si; }
            }
            if (early) {
                pdl_wait();
                pdl_launch_dependents();
            }
            for (int it = 0, kc = 0; it < npre; ++it) {
                load_h(it, kc);
                if (++kc == nk) kc = 0;
            }
            for (int it = npre, si = npre / nk, kc = npre % nk; it < total_it; ++it) {
                load_w(it, si, kc);
                load_h(it, kc);
                if (++kc == nk) { kc = 0; ++si; }
            }
        } else if (early) {
            pdl_wait();
            pdl_launch_dependents();
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kM, NP, /*a_mn=*/true, /*b_mn=*/false);
            int it = 0;
            for (int si = 0; si < my_slabs; ++si) {
                const int a = si & 1;
                mbar_wait(&acc_empty[a], ((si >> 1) & 1) ^ 1, err);
                tc_fence_after();
                const uint32_t d_tmem = tmem + a * C::kAccCols;
                for (int kc = 0; kc < nk; ++kc, ++it) {
                    const int s = it % C::kStages;
                    mbar_wait(&full[s], (it / C::kStages) & 1, err);
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * C::kStageBytes);
                    const uint32_t sb = sa + kWBytes;
#pragma unroll
                    for (int k16 = 0; k16 < kHK / 16; ++k16) {
                        // A = W^T, MN-major: 8-row K groups 1024 B apart, the two
                        // 64-column halves of M 8192 B apart; 16 K rows = 2048 B.
                        const uint64_t ad = smem_desc_sw128(sa + k16 * 2048, kHK * 128, 1024);
                        // B = hidden rows, K-major: 8-row N groups 1024 B apart;
                        // 16 K elements = 32 B inside the swizzled row.
                        const uint64_t bd = smem_desc_sw128(sb + k16 * 32, 16, 1024);
                        tc_mma(d_tmem, ad, bd, idesc, (kc > 0 || k16 > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);   // stage s free once these MMAs have read it
                }
                tc_commit(&acc_full[a]);    // accumulator a complete
            }
        }
    } else {
        // ---------------- epilogue: warps 0..3, lane = vocab column ----------------
        for (int si = 0; si < my_slabs; ++si) {
            const int slab = blockIdx.x + si * gridDim.x;
            const int a = si & 1;
            mbar_wait(&acc_full[a], (si >> 1) & 1, err);
            tc_fence_after();
            const int v = slab * kM + warp * 32 + lane;
            const uint32_t taddr = tmem + ((warp * 32) << 16) + a * C::kAccCols;
            bool nan_seen = false;
#pragma unroll 1
            for (int c0 = 0; c0 < NP; c0 += 16) {
                uint32_t r[16];
                tmem_ld16_sync(taddr + c0, r);
                if (logits) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = c0 + i;
                        if (n0 + n < N && n < NP && v < V)
                            logits[static_cast<size_t>(n0 + n) * V + v] = __uint_as_float(r[i]);
                    }
                }
                if (amax) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float x = __uint_as_float(r[i]);
                        const bool valid = v < V;
                        nan_seen |= valid && n0 + c0 + i < N && x != x;
                        const uint64_t k = warp_max_key(valid ? argmax_key(argmax_okey(x), v) : 0ull);
                        if (lane == 0) keys_s[warp * NP + c0 + i] = k;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
            if (amax) {
                if (__any_sync(0xffffffffu, nan_seen) && lane == 0) raise_error(err, SV_DEVERR_NONFINITE);
                named_barrier(1, 128);   // the four epilogue warps' keys are in
                const int nrows = N - n0 < NP ? N - n0 : NP;
                for (int n = threadIdx.x; n < nrows; n += 128) {
                    uint64_t k = keys_s[n];
#pragma unroll
                    for (int w = 1; w < 4; ++w) k = keys_s[w * NP + n] > k ? keys_s[w * NP + n] : k;
                    amax[static_cast<size_t>(n0 + n) * nslab + slab] = k;
                }
                named_barrier(1, 128);   // keys read before the next slab writes them
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int NP>
cudaError_t launch_tc(const uint16_t* hid, const uint16_t* W, float* logits, uint64_t* amax, int N, int H, int V,
                      int n0, bool w_ready, cudaStream_t st) {
    using C = TcCfg<NP>;
    alignas(64) uint8_t tmW[128], tmH[128];
    if (!encode_tmap_2d_bf16(tmW, W, V, H, static_cast<uint64_t>(V) * 2, 64, kHK)) return cudaErrorInvalidValue;
    if (!encode_tmap_2d_bf16(tmH, hid, H, N, static_cast<uint64_t>(H) * 2, kHK, NP)) return cudaErrorInvalidValue;
    static PerDeviceOnce attr_once;
    const cudaError_t ea = attr_once.run([]() {
        return cudaFuncSetAttribute(lm_head_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    });
    if (ea != cudaSuccess) return ea;
    const int nslab = (V + kM - 1) / kM;
    int grid = device_sm_count();
    if (grid > nslab) grid = nslab;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lm_head_tc_kernel<NP>, *reinterpret_cast<const CUtensorMap*>(tmW),
                              *reinterpret_cast<const CUtensorMap*>(tmH), logits, amax, N, H, V, n0, nslab,
                              w_ready ? 1 : 0, device_error_word());
}

}  // namespace

// Rows n0 .. n0+rows-1 of the pass (17 <= rows <= 256 after padding to 16).
cudaError_t launch_lm_head_tc(const uint16_t* hid, const uint16_t* W, float* logits, uint64_t* amax, int N, int H,
                              int V, int n0, int rows, bool w_ready, cudaStream_t st) {
    const int np = (rows + 15) / 16 * 16;
    switch (np) {
        case 16: return launch_tc<16>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 32: return launch_tc<32>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 48: return launch_tc<48>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 64: return launch_tc<64>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 80: return launch_tc<80>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 96: return launch_tc<96>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 112: return launch_tc<112>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 128: return launch_tc<128>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 144: return launch_tc<144>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 160: return launch_tc<160>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 176: return launch_tc<176>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 192: return launch_tc<192>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 208: return launch_tc<208>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 224: return launch_tc<224>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        case 240: return launch_tc<240>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
        default: return launch_tc<256>(hid, W, logits, amax, N, H, V, n0, w_ready, st);
    }
}

}  // namespace sv
