// hessian.cu — the Hessian accumulator: S += X^T X over token batches, H = 2 S / n
// (GPTQ guide page, "How it works" and "Source code", `_hessian_inverse_chol`; GPTQ's
// error-compensation loop page: H = 2 X^T X / N).
//
// bf16 X runs on the 5th-generation tensor cores:
//   - X (n, d) row-major is read by TMA in 64-channel x 64-token boxes with the 128-byte
//     swizzle; both GEMM operands come from the same token-major X, so both are MN-major
//     (K = tokens is the strided dimension) and the smem image is exactly the canonical
//     MN-major SW128 layout tcgen05.mma consumes.
//   - Only tiles touching the upper triangle i <= j are computed: 128 x 256 output tiles
//     (one tcgen05.mma 128x256x16 per 16 tokens), listed once per accumulator.
//   - Work units are (tile, token split); a persistent grid of one CTA per SM walks them
//     split-major so concurrently running CTAs stream the same token range (X is re-read
//     from L2, not HBM). The tiles are listed in 2D blocks of kWaveRows x kWaveCols tiles,
//     so the tiles of one wave of CTAs read only ~kWaveRows*128 + kWaveCols*256 channels
//     of each token (on a 14336-wide input X is read from HBM ~1.6x less than with the
//     tiles listed column by column; 1-2.5% faster). Splits short enough for a split's X
//     slab to stay in L2 were measured slower: their extra atomic flushes into S cost more
//     than the re-reads they save.
//   - Warp roles: warp 0 issues TMA, warp 1 issues MMA (one thread), warps 2..9 drain the
//     accumulator. TMEM holds two 128x256 fp32 accumulators (all 512 columns); every
//     1024 tokens the MMA warp switches buffers and the epilogue warps add the finished
//     buffer into fp32 registers (128 per thread), so the tensor-core accumulation chain
//     stays 1024 tokens long while a unit covers many thousands.
//   - At the end of a unit the registers are added into S with vector atomics.
// fp32 X (and bf16 X whose row stride or base does not meet TMA's 16-byte rules) runs on
// a SIMT FFMA kernel with the same upper-tile structure.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"

struct gptq_hessian {
    int64_t d;
    int device;
    int sms;
    float* S;        // d x d, row-major; the upper triangle (i <= j) is maintained
    int* status;     // device status word
    int2* tiles;     // (bi, bj) of the 128 x 256 tiles that touch the upper triangle
    int ntiles;
    int64_t n;       // tokens accumulated so far
};

namespace gptq {

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return kSMs;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return kSMs;
    return n > 0 ? n : kSMs;
}

namespace {

// ------------------------------------------------------------------------------------
// tensor-core SYRK
// ------------------------------------------------------------------------------------
constexpr int TC_BM = 128;            // output tile rows (channels i)
constexpr int TC_BN = 256;            // output tile cols (channels j)
constexpr int TC_BK = 64;             // tokens per pipeline stage
constexpr int TC_STAGES = 4;
constexpr int TC_FLUSH = 16;          // stages per TMEM accumulation chain (1024 tokens)
constexpr int TC_THREADS = 320;       // 10 warps
constexpr int TC_BOX_BYTES = 64 * TC_BK * 2;              // one 64-channel x 64-token box
constexpr int TC_A_BYTES = (TC_BM / 64) * TC_BOX_BYTES;   // 16 KB
constexpr int TC_B_BYTES = (TC_BN / 64) * TC_BOX_BYTES;   // 32 KB
constexpr int TC_STAGE_BYTES = TC_A_BYTES + TC_B_BYTES;   // 48 KB
constexpr int TC_SMEM = TC_STAGES * TC_STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t TC_IDESC = idesc_bf16_f32_mn_mn(TC_BM, TC_BN);
constexpr uint32_t TC_TMEM_COLS = 512;
// the tile order's 2D blocks: about one wave of 152 CTAs (19 x 128 + 8 x 256 channels)
constexpr int64_t kWaveRows = 19, kWaveCols = 8;

struct TcParams {
    int64_t d;
    int64_t n;
    int64_t split_tokens;  // multiple of TC_BK
    int ntiles;
    int nsplit;
    const int2* tiles;
    float* S;
    int* status;
};

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, int* status) {
    // bounded wait that ignores the abort flag: used only to let in-flight async work land
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            set_status(status, GPTQ_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__global__ void __launch_bounds__(TC_THREADS, 1) hessian_tc_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                   const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TC_STAGES * TC_STAGE_BYTES);
    // bars: full[4], empty[4], tfull[2], tempty[2], drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 17);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (TC_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * TC_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * TC_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * TC_STAGES + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 8);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tmap);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TC_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int nunits = p.ntiles * p.nsplit;

    if (warp == 0) {
        // ------------------------------- TMA producer -------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
                const int2 t = p.tiles[u % p.ntiles];
                const int64_t tok0 = (int64_t)(u / p.ntiles) * p.split_tokens;
                const int64_t tok1 = min(p.n, tok0 + p.split_tokens);
                const int nst = tok1 > tok0 ? (int)((tok1 - tok0 + TC_BK - 1) / TC_BK) : 0;
                const int i0 = t.x * TC_BM, j0 = t.y * TC_BN;
                for (int s = 0; s < nst; ++s) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full_bar(stage), TC_STAGE_BYTES);
                    const int y = (int)(tok0 + (int64_t)s * TC_BK);
                    const uint32_t sa = sbase + stage * TC_STAGE_BYTES;
#pragma unroll
                    for (int a = 0; a < TC_BM / 64; ++a)
                        tma_load_2d(sa + a * TC_BOX_BYTES, &tmap, full_bar(stage), i0 + 64 * a, y);
#pragma unroll
                    for (int b = 0; b < TC_BN / 64; ++b)
                        tma_load_2d(sa + TC_A_BYTES + b * TC_BOX_BYTES, &tmap, full_bar(stage), j0 + 64 * b, y);
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == TC_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // let every copy this thread issued land before the CTA can exit
            for (int s = 0; s < TC_STAGES; ++s)
                if (issued & (1u << s)) wait_drain(full_bar(s), (issued_par >> s) & 1u, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer ---------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int abuf = 0;
            uint32_t aphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
                const int64_t tok0 = (int64_t)(u / p.ntiles) * p.split_tokens;
                const int64_t tok1 = min(p.n, tok0 + p.split_tokens);
                const int nst = tok1 > tok0 ? (int)((tok1 - tok0 + TC_BK - 1) / TC_BK) : 0;
                for (int f0 = 0; f0 < nst && ok; f0 += TC_FLUSH) {
                    if (!mbar_wait(tempty_bar(abuf), aphase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem_base + (uint32_t)(abuf * TC_BN);
                    const int f1 = min(nst, f0 + TC_FLUSH);
                    for (int s = f0; s < f1; ++s) {
                        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = sbase + stage * TC_STAGE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < TC_BK / 16; ++kk) {
                            // 16 tokens = two 8-row swizzle atoms = 2048 bytes along K
                            const uint64_t ad = smem_desc(sa + kk * 2048, TC_BOX_BYTES, 1024, kSwizzle128B);
                            const uint64_t bd = smem_desc(sa + TC_A_BYTES + kk * 2048, TC_BOX_BYTES, 1024,
                                                          kSwizzle128B);
                            umma_f16(dt, ad, bd, TC_IDESC, (s > f0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(empty_bar(stage));
                        if (++stage == TC_STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(tfull_bar(abuf));
                    if (++abuf == 2) {
                        abuf = 0;
                        aphase ^= 1u;
                    }
                }
            }
            // every MMA issued above has completed once this arrives
            umma_commit(drain_bar);
            wait_drain(drain_bar, 0, p.status);
        }
    } else {
        // ------------------------------- epilogue (8 warps) -------------------------
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int h = (warp - 2) >> 2;   // which 128-column half of the 256-column tile
        const int64_t d = p.d;
        int abuf = 0;
        uint32_t aphase = 0;
        bool ok = true;
        float acc[128];
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
            const int2 t = p.tiles[u % p.ntiles];
            const int64_t tok0 = (int64_t)(u / p.ntiles) * p.split_tokens;
            const int64_t tok1 = min(p.n, tok0 + p.split_tokens);
            const int nst = tok1 > tok0 ? (int)((tok1 - tok0 + TC_BK - 1) / TC_BK) : 0;
            if (nst == 0) continue;
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
            for (int f0 = 0; f0 < nst; f0 += TC_FLUSH) {
                // all 32 lanes agree before the warp-collective tcgen05.ld below
                ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(abuf), aphase, abort_flag, p.status));
                if (!ok) break;
                tc_fence_after();
                const uint32_t ta = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(abuf * TC_BN + 128 * h);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(ta + 32 * c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[32 * c + i] += __uint_as_float(v[i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(abuf));
                if (++abuf == 2) {
                    abuf = 0;
                    aphase ^= 1u;
                }
            }
            if (!ok) break;
            const int64_t gi = (int64_t)t.x * TC_BM + 32 * q + lane;
            const int64_t gj0 = (int64_t)t.y * TC_BN + 128 * h;
            if (gi < d) {
                float* row = p.S + gi * d;
                if ((d & 3) == 0) {
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const int64_t gj = gj0 + 4 * m;
                        if (gj < d && gj + 3 >= gi)
                            atomicAdd(reinterpret_cast<float4*>(row + gj),
                                      make_float4(acc[4 * m], acc[4 * m + 1], acc[4 * m + 2], acc[4 * m + 3]));
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < 128; ++m) {
                        const int64_t gj = gj0 + m;
                        if (gj < d && gj >= gi) atomicAdd(row + gj, acc[m]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TC_TMEM_COLS);
    }
}

// ------------------------------------------------------------------------------------
// SIMT SYRK (fp32 X, or bf16 X that TMA cannot address): 64 x 64 upper tiles, 4 x 4 per
// thread, 32 tokens per shared-memory chunk, fp32 FFMA; splits over tokens add into S
// with atomics.
// ------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__global__ void __launch_bounds__(256) hessian_simt_kernel(const T* __restrict__ X, int64_t ld, int64_t n, int64_t d,
                                                          int64_t split_tokens, float* __restrict__ S) {
    const int nb = (int)((d + 63) / 64);
    const int bi = blockIdx.x / nb, bj = blockIdx.x % nb;
    if (bj < bi) return;
    const int64_t i0 = (int64_t)bi * 64, j0 = (int64_t)bj * 64;
    const int64_t t_begin = (int64_t)blockIdx.y * split_tokens;
    const int64_t t_end = min(n, t_begin + split_tokens);
    __shared__ float Xa[32][64 + 4];
    __shared__ float Xb[32][64 + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int64_t t0 = t_begin; t0 < t_end; t0 += 32) {
        for (int idx = threadIdx.x; idx < 32 * 64; idx += 256) {
            const int r = idx >> 6, c = idx & 63;
            const int64_t t = t0 + r;
            const bool tin = t < t_end;
            Xa[r][c] = (tin && i0 + c < d) ? to_f<T>(X[t * ld + i0 + c]) : 0.0f;
            Xb[r][c] = (tin && j0 + c < d) ? to_f<T>(X[t * ld + j0 + c]) : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int r = 0; r < 32; ++r) {
            float a[4], b[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                a[k] = Xa[r][ty * 4 + k];
                b[k] = Xb[r][tx * 4 + k];
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int64_t gi = i0 + ty * 4 + x;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int64_t gj = j0 + tx * 4 + y;
            if (gi < d && gj < d && gj >= gi) atomicAdd(S + gi * d + gj, acc[x][y]);
        }
    }
}

// H[i][j] = scale * S[min(i,j)][max(i,j)], diag_xtx[j] = S[j][j]
// H = scale * S (both triangles from S's upper one), diag = diag(S). A diagonal entry that
// is not finite (a NaN or an infinity anywhere in the accumulated X makes its channel's
// S[j][j] one) records GPTQ_ERR_NONFINITE.
__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ S, int64_t d, float scale,
                                                      float* __restrict__ H, float* __restrict__ diag,
                                                      int* __restrict__ status) {
    __shared__ float T[32][33];
    const int ti = blockIdx.y, tj = blockIdx.x;
    const int lo = min(ti, tj), hi = max(ti, tj);
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8) {
        const int64_t gi = (int64_t)lo * 32 + r, gj = (int64_t)hi * 32 + tx;
        T[r][tx] = (gi < d && gj < d) ? S[gi * d + gj] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int64_t gi = (int64_t)ti * 32 + r, gj = (int64_t)tj * 32 + tx;
        if (gi >= d || gj >= d) continue;
        float v;
        if (ti < tj) v = T[r][tx];
        else if (ti > tj) v = T[tx][r];
        else v = (r <= tx) ? T[r][tx] : T[tx][r];
        H[gi * d + gj] = scale * v;
        if (gi == gj) {
            if (diag) diag[gi] = v;
            if (!isfinite(v)) set_status(status, GPTQ_ERR_NONFINITE);
        }
    }
}

// The same on 64 x 64 tiles with 16-byte accesses (d % 4 == 0, 16-byte aligned S and H):
// upper tiles are scaled copies; a lower or diagonal tile stages its mirror tile of S
// (rows j, columns i: S's upper triangle) in shared memory and writes it transposed.
__global__ void __launch_bounds__(256) finalize4_kernel(const float* __restrict__ S, int64_t d, float scale,
                                                       float* __restrict__ H, float* __restrict__ diag,
                                                       int* __restrict__ status) {
    __shared__ float T[64][65];
    const int ti = blockIdx.y, tj = blockIdx.x;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // 16 groups of four per row, 16 rows per pass
    const int64_t i0 = (int64_t)ti * 64, j0 = (int64_t)tj * 64;
    if (ti < tj) {
        for (int r = ty; r < 64; r += 16) {
            const int64_t gi = i0 + r, gj = j0 + 4 * tx;
            if (gi >= d || gj >= d) continue;
            const float4 v = *reinterpret_cast<const float4*>(S + gi * d + gj);
            *reinterpret_cast<float4*>(H + gi * d + gj) = make_float4(scale * v.x, scale * v.y, scale * v.z, scale * v.w);
        }
        return;
    }
    // T[r][c] = S[j0 + r][i0 + c]
    for (int r = ty; r < 64; r += 16) {
        const int64_t gr = j0 + r, gc = i0 + 4 * tx;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (gr < d && gc < d) v = *reinterpret_cast<const float4*>(S + gr * d + gc);
        T[r][4 * tx] = v.x;
        T[r][4 * tx + 1] = v.y;
        T[r][4 * tx + 2] = v.z;
        T[r][4 * tx + 3] = v.w;
    }
    __syncthreads();
    for (int r = ty; r < 64; r += 16) {
        const int64_t gi = i0 + r, gj = j0 + 4 * tx;
        if (gi >= d || gj >= d) continue;
        float o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 4 * tx + e;
            // below the diagonal: S[gj + e][gi] = T[c][r]; on a diagonal tile at or above it:
            // S[gi][gj + e] = T[r][c]
            o[e] = (ti > tj || c < r) ? T[c][r] : T[r][c];
            if (ti == tj && c == r) {
                const float v = T[r][r];
                if (diag) diag[gi] = v;
                if (!isfinite(v)) set_status(status, GPTQ_ERR_NONFINITE);
            }
        }
        *reinterpret_cast<float4*>(H + gi * d + gj) = make_float4(scale * o[0], scale * o[1], scale * o[2], scale * o[3]);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

int accumulate_tc(gptq_hessian* h, const void* X, int64_t n, int64_t ld, cudaStream_t s) {
    auto enc = encode_fn();
    if (!enc) return GPTQ_ERR_CUDA;
    CUtensorMap tmap;
    cuuint64_t dims[2] = {(cuuint64_t)h->d, (cuuint64_t)n};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {64, (cuuint32_t)TC_BK};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return GPTQ_ERR_CUDA;

    // token splits: balance (tiles x splits) over the SMs, splits of >= 2048 tokens
    const int T = h->ntiles, sms = h->sms;
    int best_ks = 1;
    double best_eff = 0.0;
    for (int ks = 1; ks <= 64; ++ks) {
        if (ks > 1 && n / ks < 2048) break;
        const int64_t units = (int64_t)T * ks;
        const int64_t waves = (units + sms - 1) / sms;
        const double eff = (double)units / (double)(waves * sms);
        if (eff > best_eff + 0.01) {
            best_eff = eff;
            best_ks = ks;
        }
    }
    int64_t split = ceil_div(ceil_div(n, best_ks), TC_BK) * TC_BK;
    const int nsplit = (int)ceil_div(n, split);

    TcParams p;
    p.d = h->d;
    p.n = n;
    p.split_tokens = split;
    p.ntiles = T;
    p.nsplit = nsplit;
    p.tiles = h->tiles;
    p.S = h->S;
    p.status = h->status;
    const int units = T * nsplit;
    const int grid = std::min(units, sms);
    GPTQ_CUDA_TRY(cudaFuncSetAttribute(hessian_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM));
    GPTQ_LAUNCH(K_HESS_TC, s, hessian_tc_kernel<<<grid, TC_THREADS, TC_SMEM, s>>>(tmap, p));
    GPTQ_LAUNCH_CHECK();
    return GPTQ_OK;
}

template <typename T>
int accumulate_simt(gptq_hessian* h, const T* X, int64_t n, int64_t ld, cudaStream_t s) {
    const int64_t nb = ceil_div(h->d, 64);
    const int64_t tiles = nb * (nb + 1) / 2;
    int64_t ks = std::max<int64_t>(1, std::min<int64_t>(ceil_div(2 * h->sms, tiles), ceil_div(n, 256)));
    ks = std::min<int64_t>(ks, 65535);
    const int64_t split = ceil_div(ceil_div(n, ks), 32) * 32;
    const int64_t nsplit = ceil_div(n, split);
    dim3 grid((unsigned)(nb * nb), (unsigned)nsplit);
    GPTQ_LAUNCH(K_HESS_SIMT, s, hessian_simt_kernel<T><<<grid, 256, 0, s>>>(X, ld, n, h->d, split, h->S));
    GPTQ_LAUNCH_CHECK();
    return GPTQ_OK;
}

}  // namespace
}  // namespace gptq

using namespace gptq;

extern "C" int gptq_hessian_create(int64_t d, gptq_hessian** out) {
    if (!out || d < 1 || d > (1 << 20)) return GPTQ_ERR_INVALID_ARG;
    *out = nullptr;
    gptq_hessian* h = new gptq_hessian();
    h->d = d;
    h->n = 0;
    GPTQ_CUDA_TRY(cudaGetDevice(&h->device));
    h->sms = device_sm_count();
    // the upper tiles in 2D blocks of kWaveRows x kWaveCols tiles (block rows of a block
    // column first), so that consecutive units - the ones a wave of CTAs runs together -
    // share their channel panels
    std::vector<int2> tiles;
    const int64_t nbi = ceil_div(d, TC_BM), nbj = ceil_div(d, TC_BN);
    for (int64_t BJ = 0; BJ < nbj; BJ += kWaveCols)
        for (int64_t BI = 0; BI < nbi; BI += kWaveRows)
            for (int64_t bj = BJ; bj < std::min(nbj, BJ + kWaveCols); ++bj)
                for (int64_t bi = BI; bi < std::min(nbi, BI + kWaveRows); ++bi)
                    if (bj * TC_BN + TC_BN - 1 >= bi * TC_BM) tiles.push_back(make_int2((int)bi, (int)bj));
    h->ntiles = (int)tiles.size();
    cudaError_t e = cudaMalloc(&h->S, sizeof(float) * d * d);
    if (e == cudaSuccess) e = cudaMalloc(&h->status, sizeof(int));
    if (e == cudaSuccess) e = cudaMalloc(&h->tiles, sizeof(int2) * tiles.size());
    if (e == cudaSuccess) e = cudaMemcpy(h->tiles, tiles.data(), sizeof(int2) * tiles.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(h->S, 0, sizeof(float) * d * d);
    if (e == cudaSuccess) e = cudaMemset(h->status, 0, sizeof(int));
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        cudaFree(h->S);
        cudaFree(h->status);
        cudaFree(h->tiles);
        delete h;
        return GPTQ_ERR_CUDA;
    }
    *out = h;
    return GPTQ_OK;
}

extern "C" int gptq_hessian_reset(gptq_hessian* h, void* stream) {
    if (!h) return GPTQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GPTQ_CUDA_TRY(cudaMemsetAsync(h->S, 0, sizeof(float) * h->d * h->d, s));
    GPTQ_CUDA_TRY(cudaMemsetAsync(h->status, 0, sizeof(int), s));
    h->n = 0;
    return GPTQ_OK;
}

extern "C" int gptq_hessian_accumulate(gptq_hessian* h, const void* X, int dtype, int64_t n_tokens, int64_t ld,
                                       void* stream) {
    if (!h || n_tokens < 0 || ld < h->d) return GPTQ_ERR_INVALID_ARG;
    if (dtype != GPTQ_BF16 && dtype != GPTQ_F32) return GPTQ_ERR_INVALID_ARG;
    if (n_tokens == 0) return GPTQ_OK;
    if (!X || n_tokens > (int64_t)INT32_MAX) return GPTQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc;
    if (dtype == GPTQ_BF16) {
        const bool tma_ok = (reinterpret_cast<uintptr_t>(X) % 16 == 0) && ((ld * 2) % 16 == 0);
        rc = tma_ok ? accumulate_tc(h, X, n_tokens, ld, s)
                    : accumulate_simt<__nv_bfloat16>(h, static_cast<const __nv_bfloat16*>(X), n_tokens, ld, s);
    } else {
        rc = accumulate_simt<float>(h, static_cast<const float*>(X), n_tokens, ld, s);
    }
    if (rc == GPTQ_OK) h->n += n_tokens;
    return rc;
}

extern "C" int gptq_hessian_finalize(gptq_hessian* h, float* H, float* diag_xtx, int64_t* n_tokens, void* stream) {
    if (!h || !H) return GPTQ_ERR_INVALID_ARG;
    if (h->n <= 0) return GPTQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float scale = (float)(2.0 / (double)h->n);
    if (h->d % 4 == 0 && ((reinterpret_cast<uintptr_t>(H) | reinterpret_cast<uintptr_t>(h->S)) % 16 == 0)) {
        const unsigned nt = (unsigned)ceil_div(h->d, 64);
        GPTQ_LAUNCH(K_FINALIZE, s, finalize4_kernel<<<dim3(nt, nt), 256, 0, s>>>(h->S, h->d, scale, H, diag_xtx,
                                                                                     h->status));
    } else {
        const unsigned nt = (unsigned)ceil_div(h->d, 32);
        GPTQ_LAUNCH(K_FINALIZE, s, finalize_kernel<<<dim3(nt, nt), 256, 0, s>>>(h->S, h->d, scale, H, diag_xtx,
                                                                                    h->status));
    }
    GPTQ_LAUNCH_CHECK();
    if (n_tokens) *n_tokens = h->n;
    return finish_call(h->status, s);
}

extern "C" int gptq_hessian_destroy(gptq_hessian* h) {
    if (!h) return GPTQ_ERR_INVALID_ARG;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->S);
    cudaFree(h->status);
    cudaFree(h->tiles);
    cudaSetDevice(dev);
    (void)cudaGetLastError();
    delete h;
    return GPTQ_OK;
}

namespace gptq {
// this file's copy of the pipeline-wait limit (the library's test hook sets every copy)
cudaError_t hessian_set_wait_limit(unsigned long long ns) { return set_pipeline_wait_limit_this_unit(ns); }
}  // namespace gptq
