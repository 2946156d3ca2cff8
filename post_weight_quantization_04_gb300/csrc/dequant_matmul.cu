// dequant_matmul.cu — Y = X Wq^T computed straight from GPTQ's stored form: packed
// b-bit codes, per-group scales and zero points, and the column-to-group index g_idx.
//
// Wq[o][k] = s[o][g] * (u[o][k] - z[o][g]) with g = g_idx[k] (GPTQ guide page, "When it
// breaks": with act_order, a kernel that consumes groups needs the stored column-to-group
// index; AutoGPTQ page, `dequantize_weight`: scale * (code - zero)). u is the k-th b-bit
// field of row o's LSB-first bitstream (the packing of `gptq_pack`).
//
// Structure (one CTA per SM, persistent over a contiguous range of 128 tokens x 128
// outputs tiles, output tile major):
//   warp 0       TMA producer: the 128 x 64 bf16 X box of each K step (128-byte swizzle)
//   warp 1       single-thread tcgen05.mma issuer, kind::f16 (bf16 x bf16 -> fp32),
//                M = N = 128, K = 16 per instruction, two TMEM accumulators
//   warps 2..5   epilogue: TMEM -> registers -> fp32 Y
//   warps 6..13  dequantisers: unpack the b-bit codes of 128 output rows x 64 columns,
//                look up s and z through g_idx (per-tile tables in shared memory), and
//                write the bf16 weights straight into the K-major, 128-byte-swizzled image
//                the MMA reads
//   warp 14      loader: the packed words of each K step into a shared ring by cp.async
//                (so the dequantisers, which must fence their writes for the tensor core,
//                never have a global load in flight)
// The weight tile is produced on chip, so W is read from HBM as b bits per weight.
// Every mbarrier wait is bounded (GPTQ_ERR_TIMEOUT into the status word, then unwind).
#include <cuda_bf16.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "tc_gemm.cuh"

namespace gptq {

namespace {

constexpr int D_BM = 128, D_BN = 128, D_BK = 64;
// X boxes come from L2 or HBM and need a deep ring to hide their latency; the weight
// boxes are produced on chip and need only a short one
constexpr int D_XS = 3, D_WS = 3, D_PS = 4;
constexpr int D_BOX = D_BM * D_BK * 2;       // 16 KB: 128 rows x 64 bf16
constexpr int D_PBOX = D_BN * 32;               // one K step of packed words: 128 rows x <= 32 B
constexpr int D_RING = (D_XS + D_WS) * D_BOX + D_PS * D_PBOX;  // X ring, weight ring, packed ring
constexpr int D_DQ_WARPS = 8;
constexpr int D_LOADER_WARP = 6 + D_DQ_WARPS;
constexpr int D_THREADS = 32 * (7 + D_DQ_WARPS);
constexpr int D_SMEM_MAX = 227 * 1024;
constexpr uint32_t D_TMEM_COLS = 2 * D_BN;
// kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (1), both K-major, N >> 3, M >> 4
constexpr uint32_t D_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(D_BN >> 3) << 17) |
                             ((uint32_t)(D_BM >> 4) << 24);

struct DParams {
    int T, N, K;
    int tiles_n, ntiles;
    const uint32_t* packed;
    int64_t words;  // 32-bit words per packed row
    const float* scales;
    const uint8_t* zeros;
    int64_t G;
    const int32_t* g_idx;
    void* Y;          // fp32, or bf16 with GPTQ_DQ_BF16_OUT
    int64_t ldy;
    int relu, bf16_out;
    int* status;
    // shared-memory layout after the stages and barriers: g_idx as int16 (K entries), then
    // (when tab) the tile's scales (128 x sp floats) and zero points (128 x zp bytes); sp
    // odd and zp / 4 odd so the 32 rows a warp reads hit 32 different banks
    int tab, sp, zp;
    int g_off, s_off, z_off;
    int gs;           // the grouped kernel's group size in columns; for the general kernel the
                      // group size of the grouped kernel launched with it, 0 if none was
};

// Whether every column's group is g_idx[k] == k / gs (contiguous groups of gs columns), as
// the whole CTA sees it. Both kernels of a call decide with the same test, so exactly one
// of them does the work; the other returns before touching shared memory or TMEM.
__device__ __forceinline__ bool cta_groups_contiguous(const int32_t* __restrict__ g_idx, int K, int gs) {
    int bad = 0;
    for (int k = threadIdx.x; k < K; k += blockDim.x) bad |= (g_idx[k] != k / gs) ? 1 : 0;
    return __syncthreads_or(bad) == 0;
}

// Named barrier ID over N threads that also ANDs a predicate across them: a group of warps
// that shares a named barrier inside its tile loop leaves the loop together (a warp whose
// bounded wait gave up must not leave the others waiting at that barrier).
template <int ID, int N>
__device__ __forceinline__ bool bar_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "barrier.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)(v ? 1 : 0)), "n"(ID), "n"(N)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half), .y = b
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            set_status(status, GPTQ_ERR_TIMEOUT);
            return;
        }
    }
}

// TAB: scales and zero points come from the per-tile tables in shared memory (a compile-time
// choice: with a runtime flag the compiler may issue both sources' loads)
template <int BITS, bool TAB>
__global__ void __launch_bounds__(D_THREADS, 1) dequant_matmul_kernel(const __grid_constant__ CUtensorMap tX,
                                                                     const DParams p) {
    if (p.gs > 0 && cta_groups_contiguous(p.g_idx, p.K, p.gs)) return;   // the grouped kernel does the work
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + D_RING);
    int16_t* g16 = reinterpret_cast<int16_t*>(smem + p.g_off);
    float* s_tab = reinterpret_cast<float*>(smem + p.s_off);
    uint8_t* z_tab = smem + p.z_off;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 30);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 31);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem), bar0 = smem_u32(bars);
    auto xfull = [&](int s) { return bar0 + 8u * s; };                     // X box landed (TMA)
    auto xempty = [&](int s) { return bar0 + 8u * (D_XS + s); };           // its MMAs are done
    auto wfull = [&](int s) { return bar0 + 8u * (2 * D_XS + s); };        // weight box written
    auto wempty = [&](int s) { return bar0 + 8u * (2 * D_XS + D_WS + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * D_XS + 2 * D_WS + 4);
    auto pfull = [&](int s) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + 5 + s); };        // words landed
    auto pempty = [&](int s) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + 5 + D_PS + s); }; // words read
    uint8_t* pring = smem + (D_XS + D_WS) * D_BOX;
    const int ktiles = p.K / D_BK;
    // each CTA walks a contiguous range of tiles, ordered by output tile first, so the
    // weight rows (and their scale table) stay the same across consecutive tiles
    const int t_begin = (int)((int64_t)blockIdx.x * p.ntiles / gridDim.x);
    const int t_end = (int)((int64_t)(blockIdx.x + 1) * p.ntiles / gridDim.x);
    const int tiles_m = p.ntiles / p.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < D_XS; ++s) {
            mbar_init(xfull(s), 1);
            mbar_init(xempty(s), 1);
        }
        for (int s = 0; s < D_WS; ++s) {
            mbar_init(wfull(s), D_DQ_WARPS);
            mbar_init(wempty(s), 1);
        }
        for (int s = 0; s < D_PS; ++s) {
            mbar_init(pfull(s), 32);            // one cp.async completion per loader lane
            mbar_init(pempty(s), D_DQ_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tX);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), D_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------- TMA producer (X) ---------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int t = t_begin; t < t_end && ok; ++t) {
                const int tm = t % tiles_m;
                for (int kt = 0; kt < ktiles; ++kt) {
                    if (!mbar_wait(xempty(stage), phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(xfull(stage), D_BOX);
                    tma_load_2d(sbase + stage * D_BOX, &tX, xfull(stage), kt * D_BK, tm * D_BM);
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == D_XS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < D_XS; ++s)
                if (issued & (1u << s)) drain(xfull(s), (issued_par >> s) & 1u, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer ---------------------------------
        if (lane == 0) {
            int xs = 0, ws = 0, abuf = 0;
            uint32_t xph = 0, wph = 0, aphase = 0;
            bool ok = true;
            for (int t = t_begin; t < t_end && ok; ++t) {
                if (!mbar_wait(tempty(abuf), aphase ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(abuf * D_BN);
                for (int kt = 0; kt < ktiles; ++kt) {
                    if (!mbar_wait(xfull(xs), xph, abort_flag, p.status) ||
                        !mbar_wait(wfull(ws), wph, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + xs * D_BOX, sb = sbase + (D_XS + ws) * D_BOX;
#pragma unroll
                    for (int kk = 0; kk < D_BK / 16; ++kk) {
                        // 16 bf16 = 32 bytes along K inside the 128-byte swizzle row
                        const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024, kSwizzle128B);
                        umma_f16(dt, ad, bd, D_IDESC, (kt > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(xempty(xs));
                    umma_commit(wempty(ws));
                    if (++xs == D_XS) {
                        xs = 0;
                        xph ^= 1u;
                    }
                    if (++ws == D_WS) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull(abuf));
                if (++abuf == 2) {
                    abuf = 0;
                    aphase ^= 1u;
                }
            }
            umma_commit(drain_bar);
            drain(drain_bar, 0, p.status);
        }
    } else if (warp < 6) {
        // ------------------------------- epilogue (4 warps) -------------------------
        const int q = warp & 3;
        int abuf = 0;
        uint32_t aphase = 0;
        const bool vec = ((p.ldy & 7) == 0) && ((reinterpret_cast<uintptr_t>(p.Y) & 15) == 0);
        for (int t = t_begin; t < t_end; ++t) {
            const int tm = t % tiles_m, tn = t / tiles_m;
            if (!mbar_wait_warp(tfull(abuf), aphase, abort_flag, p.status)) break;
            tc_fence_after();
            const int row = tm * D_BM + 32 * q + lane;
            const uint32_t ta = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(abuf * D_BN);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(ta + 32 * c, v);
                tmem_ld_wait();
                const int col = tn * D_BN + 32 * c;
                float f[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) f[jj] = p.relu ? fmaxf(__uint_as_float(v[jj]), 0.0f) : __uint_as_float(v[jj]);
                if (row < p.T && p.bf16_out) {
                    __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.Y) + (int64_t)row * p.ldy + col;
                    if (vec && col + 32 <= p.N) {
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            reinterpret_cast<uint4*>(y)[jj] =
                                make_uint4(bf16x2(f[8 * jj], f[8 * jj + 1]), bf16x2(f[8 * jj + 2], f[8 * jj + 3]),
                                           bf16x2(f[8 * jj + 4], f[8 * jj + 5]), bf16x2(f[8 * jj + 6], f[8 * jj + 7]));
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            if (col + jj < p.N) y[jj] = __float2bfloat16_rn(f[jj]);
                    }
                } else if (row < p.T) {
                    float* y = reinterpret_cast<float*>(p.Y) + (int64_t)row * p.ldy + col;
                    if (vec && col + 32 <= p.N) {
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            reinterpret_cast<float4*>(y)[jj] = make_float4(f[4 * jj], f[4 * jj + 1], f[4 * jj + 2], f[4 * jj + 3]);
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj)
                            if (col + jj < p.N) y[jj] = f[jj];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(abuf));
            if (++abuf == 2) {
                abuf = 0;
                aphase ^= 1u;
            }
        }
    } else if (warp == D_LOADER_WARP) {
        // ------------------------------- packed-word loader -------------------------
        // Copies each K step's packed words (128 rows x 8*BITS bytes) into the packed ring
        // with cp.async, completion counted on pfull. The expanding warps then hold no
        // global load in flight when they fence their shared-memory writes for the
        // tensor core.
        int ps = 0;
        uint32_t pph = 0;
        bool ok = true;
        for (int t = t_begin; t < t_end && ok; ++t) {
            const int tn = t / tiles_m;
            for (int kt = 0; kt < ktiles; ++kt) {
                if (!mbar_wait_warp(pempty(ps), pph ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int r = lane + 32 * it;
                    const int o = tn * D_BN + r;
                    if (o < p.N) {
                        const uint32_t dst = smem_u32(pring + ps * D_PBOX + r * 32);
                        const uint32_t* src = p.packed + (int64_t)o * p.words + 2 * BITS * kt;
                        if (BITS == 3) {
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst + 8), "l"(src + 2) : "memory");
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst + 16), "l"(src + 4) : "memory");
                        } else {
#pragma unroll
                            for (int q = 0; q < BITS / 2; ++q)
                                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16 * q),
                                             "l"(src + 4 * q)
                                             : "memory");
                        }
                    }
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(pfull(ps)) : "memory");
                if (++ps == D_PS) {
                    ps = 0;
                    pph ^= 1u;
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ------------------------------- dequantisers (8 warps) ---------------------
        // A K step's weight box is 128 rows x 8 chunks of 8 columns. Thread i expands chunk
        // j = i % 8 of rows r = i / 8 + 32 it (it = 0..3); each chunk is one 16-byte unit of
        // the swizzled shared-memory image, and its codes are 8*BITS bits of the row's words
        // in the packed ring.
        const int i = threadIdx.x - 6 * 32;
        const int j = i & 7, rb = i >> 3;
        constexpr int NDQ = 32 * D_DQ_WARPS;
        auto dq_sync = [] { asm volatile("bar.sync 2, %0;" ::"n"(32 * D_DQ_WARPS) : "memory"); };
        // g_idx into shared memory once (validated: out-of-range groups read group 0)
        for (int k = i; k < p.K; k += NDQ) {
            int g = p.g_idx[k];
            if (g < 0 || g >= p.G) {
                set_status(p.status, GPTQ_ERR_INVALID_ARG);
                g = 0;
            }
            g16[k] = (int16_t)g;
        }
        dq_sync();
        // bits of chunk j inside the step's 2*BITS words: [8*BITS*j, 8*BITS*(j+1))
        constexpr int CB = 8 * BITS;
        const int w0 = (CB * j) >> 5, sh = (CB * j) & 31;
        const bool two = (BITS == 3) && (sh + CB > 32);   // the chunk straddles two words
        int ws = 0, ps = 0, tab_tn = -1;
        uint32_t wph = 0, pph = 0;
        bool ok = true;
        for (int t = t_begin; t < t_end; ++t) {
            // all expansion warps leave together if any of them gave up a wait; this barrier
            // also means every thread is done with the previous tile's table
            if (!bar_all<2, 32 * D_DQ_WARPS>(ok)) break;
            const int tn = t / tiles_m;
            const float* srow[4];
            const uint8_t* zrow[4];
            bool live[4];
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int o = tn * D_BN + rb + 32 * it;
                live[it] = o < p.N;
                const int64_t oo = live[it] ? o : 0;
                srow[it] = p.scales + oo * p.G;
                zrow[it] = p.zeros + oo * p.G;
            }
            if (TAB && tn != tab_tn) {
                // this tile's scales and zero points, read once, coalesced
                tab_tn = tn;
                const int64_t n = (int64_t)D_BN * p.G;
                for (int64_t idx = i; idx < n; idx += NDQ) {
                    const int rr = (int)(idx / p.G), g = (int)(idx - (int64_t)rr * p.G);
                    const int oo = tn * D_BN + rr;
                    const bool lv = oo < p.N;
                    s_tab[rr * p.sp + g] = lv ? p.scales[(int64_t)oo * p.G + g] : 0.0f;
                    z_tab[rr * p.zp + g] = lv ? p.zeros[(int64_t)oo * p.G + g] : (uint8_t)0;
                }
                dq_sync();
            }
            for (int kt = 0; kt < ktiles; ++kt) {
                if (!mbar_wait_warp(pfull(ps), pph, abort_flag, p.status) ||
                    !mbar_wait_warp(wempty(ws), wph ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                // the chunk's 8 codes of each row, least significant first
                uint32_t v[4];
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const uint32_t* wr = reinterpret_cast<const uint32_t*>(pring + ps * D_PBOX + (rb + 32 * it) * 32);
                    const uint32_t lo = wr[w0], hi = two ? wr[w0 + 1] : 0u;
                    v[it] = live[it] ? (two ? __funnelshift_r(lo, hi, sh) : (lo >> sh)) : 0u;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(pempty(ps));   // the words are in registers
                if (++ps == D_PS) {
                    ps = 0;
                    pph ^= 1u;
                }
                const int k0 = kt * D_BK + 8 * j;
                const uint4 g8 = *reinterpret_cast<const uint4*>(g16 + k0);   // the chunk's 8 groups
                const uint32_t gw[4] = {g8.x, g8.y, g8.z, g8.w};
                int gc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) gc[e] = (int)(int16_t)((gw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
                bool one_group = true;
#pragma unroll
                for (int e = 1; e < 8; ++e) one_group = one_group && gc[e] == gc[0];
                uint8_t* sbox = smem + (D_XS + ws) * D_BOX;
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int r = rb + 32 * it;
                    float s = 0.0f, zb = 8388608.0f;
                    auto look = [&](int g) {
                        if (TAB) {
                            s = s_tab[r * p.sp + g];
                            zb = 8388608.0f + (float)z_tab[r * p.zp + g];
                        } else {
                            s = live[it] ? srow[it][g] : 0.0f;
                            zb = 8388608.0f + (live[it] ? (float)zrow[it][g] : 0.0f);
                        }
                    };
                    if (one_group) look(gc[0]);
                    float wq[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (!one_group) look(gc[e]);
                        const uint32_t u = (v[it] >> (BITS * e)) & ((1u << BITS) - 1u);
                        // 2^23 + u as a float, minus 2^23 + z: u - z exactly, no conversion
                        wq[e] = s * (__uint_as_float(0x4B000000u | u) - zb);
                    }
                    // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
                    *reinterpret_cast<uint4*>(sbox + r * 128 + ((j ^ (r & 7)) << 4)) =
                        make_uint4(bf16x2(wq[0], wq[1]), bf16x2(wq[2], wq[3]), bf16x2(wq[4], wq[5]),
                                   bf16x2(wq[6], wq[7]));
                }
                fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(wfull(ws));
                if (++ws == D_WS) {
                    ws = 0;
                    wph ^= 1u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, D_TMEM_COLS);
    }
}


// ------------------------------------------------------------------------------------
// Contiguous groups (g_idx[k] = k / gs with gs a multiple of 64, no act_order): the codes
// go to the tensor cores exact. Y = sum_g s[:, g] * P_g with P_g = X[:, g] (u - z_g)^T:
// u - z is a small integer, exact in bf16, and the products X * (u - z) are exact in
// fp32, so the only rounding left is the fp32 accumulation. Each group's partial P_g goes
// to one of two TMEM buffers; the epilogue folds s[o][g] * P_g into a running total kept
// in a third TMEM buffer while the MMAs of the next group fill the other partial buffer.
// The expansion is four LOP3 / HSUB2 / PRMT triples per 8 codes: (2^7 + u) is formed as a
// bf16 bit pattern, (2^7 + z) subtracted exactly, and the pairs put in column order.
// ------------------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ uint4 codes_minus_zero(uint32_t v, uint32_t zz) {
    constexpr uint32_t LOW = (1u << (4 * BITS)) - 1u;                // codes 0..3
    const uint32_t vv = (v & LOW) | ((v >> (4 * BITS)) << 16);        // codes 4..7 -> upper half
    constexpr uint32_t M = ((1u << BITS) - 1u) * 0x00010001u;
    uint32_t t[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        // (u_e, u_{e+4}) as the bf16 pair (128 + u_e, 128 + u_{e+4})
        const uint32_t b = ((vv >> (BITS * e)) & M) | 0x43004300u;
        const __nv_bfloat162 d = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&b),
                                         *reinterpret_cast<const __nv_bfloat162*>(&zz));
        t[e] = *reinterpret_cast<const uint32_t*>(&d);
    }
    return make_uint4(__byte_perm(t[0], t[1], 0x5410), __byte_perm(t[2], t[3], 0x5410),
                      __byte_perm(t[0], t[1], 0x7632), __byte_perm(t[2], t[3], 0x7632));
}

constexpr int G_PARTS = 3;             // TMEM partials in flight (128 columns each)
// warps: producer, MMA, 8 epilogue, loader, 4 expansion (GQ_ITEMS rows each per lane)
constexpr int GQ_EPI_WARPS = 8, GQ_LOADER_WARP = 2 + GQ_EPI_WARPS, GQ_DQ_WARPS = 4;
constexpr int GQ_ITEMS = D_BN * 8 / (32 * GQ_DQ_WARPS);
constexpr int GQ_THREADS = 32 * (GQ_LOADER_WARP + 1 + GQ_DQ_WARPS);
constexpr uint32_t G_TMEM_COLS = 512;  // three partials, then the running total

template <int BITS>
__global__ void __launch_bounds__(GQ_THREADS, 1) dequant_matmul_grouped_kernel(const __grid_constant__ CUtensorMap tX,
                                                                             const DParams p) {
    if (!cta_groups_contiguous(p.g_idx, p.K, p.gs)) return;   // scattered groups: the general kernel's work
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + D_RING);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 30);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 31);
    float* s_tab = reinterpret_cast<float*>(smem + p.s_off);   // epilogue's: G groups x 128 outputs
    uint8_t* z_tab = smem + p.z_off;                            // dequantisers': 128 rows x zp groups

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem), bar0 = smem_u32(bars);
    auto xfull = [&](int s) { return bar0 + 8u * s; };
    auto xempty = [&](int s) { return bar0 + 8u * (D_XS + s); };
    auto wfull = [&](int s) { return bar0 + 8u * (2 * D_XS + s); };
    auto wempty = [&](int s) { return bar0 + 8u * (2 * D_XS + D_WS + s); };
    auto gfull = [&](int b) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + b); };                 // partial b ready
    auto gempty = [&](int b) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + G_PARTS + b); };      // partial b folded
    const uint32_t drain_bar = bar0 + 8u * (2 * D_XS + 2 * D_WS + 2 * G_PARTS);
    auto pfull = [&](int s) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + 2 * G_PARTS + 1 + s); };
    auto pempty = [&](int s) { return bar0 + 8u * (2 * D_XS + 2 * D_WS + 2 * G_PARTS + 1 + D_PS + s); };
    uint8_t* pring = smem + (D_XS + D_WS) * D_BOX;
    const int ktiles = p.K / D_BK;
    const int gsteps = p.gs / D_BK;        // K steps per group
    const int ngroups = (int)p.G;
    const int t_begin = (int)((int64_t)blockIdx.x * p.ntiles / gridDim.x);
    const int t_end = (int)((int64_t)(blockIdx.x + 1) * p.ntiles / gridDim.x);
    const int tiles_m = p.ntiles / p.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < D_XS; ++s) {
            mbar_init(xfull(s), 1);
            mbar_init(xempty(s), 1);
        }
        for (int s = 0; s < D_WS; ++s) {
            mbar_init(wfull(s), GQ_DQ_WARPS);
            mbar_init(wempty(s), 1);
        }
        for (int s = 0; s < D_PS; ++s) {
            mbar_init(pfull(s), 32);
            mbar_init(pempty(s), GQ_DQ_WARPS);
        }
        for (int b = 0; b < G_PARTS; ++b) {
            mbar_init(gfull(b), 1);
            mbar_init(gempty(b), GQ_EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tX);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), G_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------- TMA producer (X) ---------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int t = t_begin; t < t_end && ok; ++t) {
                const int tm = t % tiles_m;
                for (int kt = 0; kt < ktiles; ++kt) {
                    if (!mbar_wait(xempty(stage), phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(xfull(stage), D_BOX);
                    tma_load_2d(sbase + stage * D_BOX, &tX, xfull(stage), kt * D_BK, tm * D_BM);
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == D_XS) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < D_XS; ++s)
                if (issued & (1u << s)) drain(xfull(s), (issued_par >> s) & 1u, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer ---------------------------------
        if (lane == 0) {
            int xs = 0, ws = 0, pb = 0;
            uint32_t xph = 0, wph = 0, pph = 0;
            bool ok = true;
            for (int t = t_begin; t < t_end && ok; ++t) {
                for (int g = 0; g < ngroups && ok; ++g) {
                    if (!mbar_wait(gempty(pb), pph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem_base + (uint32_t)(pb * D_BN);
                    for (int ks = 0; ks < gsteps; ++ks) {
                        if (!mbar_wait(xfull(xs), xph, abort_flag, p.status) ||
                            !mbar_wait(wfull(ws), wph, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = sbase + xs * D_BOX, sb = sbase + (D_XS + ws) * D_BOX;
#pragma unroll
                        for (int kk = 0; kk < D_BK / 16; ++kk) {
                            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024, kSwizzle128B);
                            const uint64_t bd = smem_desc(sb + kk * 32, 16, 1024, kSwizzle128B);
                            umma_f16(dt, ad, bd, D_IDESC, (ks > 0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(xempty(xs));
                        umma_commit(wempty(ws));
                        if (++xs == D_XS) {
                            xs = 0;
                            xph ^= 1u;
                        }
                        if (++ws == D_WS) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(gfull(pb));
                    if (++pb == G_PARTS) {
                        pb = 0;
                        pph ^= 1u;
                    }
                }
            }
            umma_commit(drain_bar);
            drain(drain_bar, 0, p.status);
        }
    } else if (warp < 2 + GQ_EPI_WARPS) {
        // ------------------------------- epilogue (8 warps) -------------------------
        // row t of the tile per thread (warp % 4 picks the TMEM lane quarter), one half of
        // the 128 output columns per warp; per group: R (+)= s[o][g] * P_g chunk by chunk;
        // after the last group Y = R (relu, bf16 as asked)
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;   // 0..255
        int pb = 0, tab_tn = -1;
        uint32_t pph = 0;
        bool ok = true;
        const bool vec = ((p.ldy & 7) == 0) && ((reinterpret_cast<uintptr_t>(p.Y) & 15) == 0);
        const uint32_t lanes = (uint32_t)(32 * q) << 16;
        for (int t = t_begin; t < t_end; ++t) {
            // all epilogue warps leave together if any of them gave up a wait; this barrier
            // also means every thread is done with the previous tile's table
            if (!bar_all<3, 32 * GQ_EPI_WARPS>(ok)) break;
            const int tm = t % tiles_m, tn = t / tiles_m;
            if (tn != tab_tn) {
                // this tile's scales, [output][group], read once, coalesced
                tab_tn = tn;
                if (et < D_BN) {
                    const int o = tn * D_BN + et;   // thread et fills output et's column of the table
                    for (int g = 0; g < ngroups; ++g)
                        s_tab[g * D_BN + et] = o < p.N ? p.scales[(int64_t)o * p.G + g] : 0.0f;
                }
                asm volatile("bar.sync 3, %0;" ::"n"(32 * GQ_EPI_WARPS) : "memory");
            }
            const int row = tm * D_BM + 32 * q + lane;
            for (int g = 0; g < ngroups; ++g) {
                if (!mbar_wait_warp(gfull(pb), pph, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool first = g == 0, last = g == ngroups - 1;
#pragma unroll 1
                for (int c = 2 * half; c < 2 * half + 2; ++c) {
                    uint32_t v[32], rr[32];
                    tmem_ld_32x32b_x32(tmem_base + lanes + (uint32_t)(pb * D_BN + 32 * c), v);
                    if (!first) tmem_ld_32x32b_x32(tmem_base + lanes + (uint32_t)(G_PARTS * D_BN + 32 * c), rr);
                    tmem_ld_wait();
                    // the group's 32 scales of this chunk: the same for every row, 16-byte broadcast reads
                    const float4* sc = reinterpret_cast<const float4*>(s_tab + g * D_BN + 32 * c);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 s4 = sc[j4];
                        const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * j4 + e;
                            rr[j] = __float_as_uint(fmaf(sv[e], __uint_as_float(v[j]), first ? 0.0f : __uint_as_float(rr[j])));
                        }
                    }
                    if (!last) {
                        tmem_st_32x32b_x32(tmem_base + lanes + (uint32_t)(G_PARTS * D_BN + 32 * c), rr);
                        continue;
                    }
                    const int col = tn * D_BN + 32 * c;
                    if (p.relu) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(fmaxf(__uint_as_float(rr[j]), 0.0f));
                    }
                    if (row < p.T && p.bf16_out) {
                        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.Y) + (int64_t)row * p.ldy + col;
                        if (vec && col + 32 <= p.N) {
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj)
                                reinterpret_cast<uint4*>(y)[jj] = make_uint4(
                                    bf16x2(__uint_as_float(rr[8 * jj]), __uint_as_float(rr[8 * jj + 1])),
                                    bf16x2(__uint_as_float(rr[8 * jj + 2]), __uint_as_float(rr[8 * jj + 3])),
                                    bf16x2(__uint_as_float(rr[8 * jj + 4]), __uint_as_float(rr[8 * jj + 5])),
                                    bf16x2(__uint_as_float(rr[8 * jj + 6]), __uint_as_float(rr[8 * jj + 7])));
                        } else {
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj)
                                if (col + jj < p.N) y[jj] = __float2bfloat16_rn(__uint_as_float(rr[jj]));
                        }
                    } else if (row < p.T) {
                        float* y = reinterpret_cast<float*>(p.Y) + (int64_t)row * p.ldy + col;
                        if (vec && col + 32 <= p.N) {
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj)
                                reinterpret_cast<uint4*>(y)[jj] = make_uint4(rr[4 * jj], rr[4 * jj + 1], rr[4 * jj + 2], rr[4 * jj + 3]);
                        } else {
#pragma unroll
                            for (int jj = 0; jj < 32; ++jj)
                                if (col + jj < p.N) y[jj] = __uint_as_float(rr[jj]);
                        }
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(gempty(pb));
                if (++pb == G_PARTS) {
                    pb = 0;
                    pph ^= 1u;
                }
            }
        }
    } else if (warp == GQ_LOADER_WARP) {
        // ------------------------------- packed-word loader (as in the general kernel)
        int ps = 0;
        uint32_t pph = 0;
        bool ok = true;
        for (int t = t_begin; t < t_end && ok; ++t) {
            const int tn = t / tiles_m;
            for (int kt = 0; kt < ktiles; ++kt) {
                if (!mbar_wait_warp(pempty(ps), pph ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int r = lane + 32 * it;
                    const int o = tn * D_BN + r;
                    if (o < p.N) {
                        const uint32_t dst = smem_u32(pring + ps * D_PBOX + r * 32);
                        const uint32_t* src = p.packed + (int64_t)o * p.words + 2 * BITS * kt;
                        if (BITS == 3) {
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst + 8), "l"(src + 2) : "memory");
                            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst + 16), "l"(src + 4) : "memory");
                        } else {
#pragma unroll
                            for (int q = 0; q < BITS / 2; ++q)
                                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16 * q),
                                             "l"(src + 4 * q)
                                             : "memory");
                        }
                    }
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(pfull(ps)) : "memory");
                if (++ps == D_PS) {
                    ps = 0;
                    pph ^= 1u;
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ------------------------------- expansion (4 warps): u - z, exact ---------
        // thread i: chunk j = i % 8 of rows i / 8 + RS * it (it < GQ_ITEMS)
        const int i = threadIdx.x - 32 * (GQ_LOADER_WARP + 1);
        const int j = i & 7, rb = i >> 3;
        constexpr int NDQ = 32 * GQ_DQ_WARPS, RS = NDQ / 8;
        auto dq_sync = [] { asm volatile("bar.sync 2, %0;" ::"n"(32 * GQ_DQ_WARPS) : "memory"); };
        constexpr int CB = 8 * BITS;
        const int w0 = (CB * j) >> 5, sh = (CB * j) & 31;
        const bool two = (BITS == 3) && (sh + CB > 32);
        int ws = 0, ps = 0, tab_tn = -1;
        uint32_t wph = 0, pph = 0;
        bool ok = true;
        for (int t = t_begin; t < t_end; ++t) {
            // all expansion warps leave together if any of them gave up a wait; this barrier
            // also means every thread is done with the previous tile's table
            if (!bar_all<2, 32 * GQ_DQ_WARPS>(ok)) break;
            const int tn = t / tiles_m;
            bool live[GQ_ITEMS];
#pragma unroll
            for (int it = 0; it < GQ_ITEMS; ++it) live[it] = tn * D_BN + rb + RS * it < p.N;
            if (tn != tab_tn) {
                tab_tn = tn;
                const int64_t n = (int64_t)D_BN * p.G;
                for (int64_t idx = i; idx < n; idx += NDQ) {
                    const int rr = (int)(idx / p.G), g = (int)(idx - (int64_t)rr * p.G);
                    const int oo = tn * D_BN + rr;
                    z_tab[rr * p.zp + g] = oo < p.N ? p.zeros[(int64_t)oo * p.G + g] : (uint8_t)0;
                }
                dq_sync();
            }
            for (int kt = 0; kt < ktiles; ++kt) {
                if (!mbar_wait_warp(pfull(ps), pph, abort_flag, p.status) ||
                    !mbar_wait_warp(wempty(ws), wph ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                uint32_t v[GQ_ITEMS];
#pragma unroll
                for (int it = 0; it < GQ_ITEMS; ++it) {
                    const uint32_t* wr = reinterpret_cast<const uint32_t*>(pring + ps * D_PBOX + (rb + RS * it) * 32);
                    const uint32_t lo = wr[w0], hi = two ? wr[w0 + 1] : 0u;
                    v[it] = live[it] ? (two ? __funnelshift_r(lo, hi, sh) : (lo >> sh)) : 0u;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(pempty(ps));
                if (++ps == D_PS) {
                    ps = 0;
                    pph ^= 1u;
                }
                const int g = kt / gsteps;
                uint8_t* sbox = smem + (D_XS + ws) * D_BOX;
#pragma unroll
                for (int it = 0; it < GQ_ITEMS; ++it) {
                    const int r = rb + RS * it;
                    // rows past N: codes 0 and zero point 0 give exact zeros
                    const uint32_t z = live[it] ? (uint32_t)z_tab[r * p.zp + g] : 0u;
                    const uint32_t zz = (0x4300u | z) * 0x00010001u;
                    *reinterpret_cast<uint4*>(sbox + r * 128 + ((j ^ (r & 7)) << 4)) = codes_minus_zero<BITS>(v[it], zz);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(wfull(ws));
                if (++ws == D_WS) {
                    ws = 0;
                    wph ^= 1u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, G_TMEM_COLS);
    }
}

}  // namespace
}  // namespace gptq

using namespace gptq;

extern "C" int gptq_dequant_matmul(const void* X, int64_t T, int64_t K, int64_t ldx, const uint32_t* packed,
                                   const float* scales, const uint8_t* zeros, const int32_t* g_idx, int64_t N,
                                   int64_t G, int bits, int flags, void* Y, int64_t ldy, void* stream) {
    if (T < 0 || K < 0 || N < 0) return GPTQ_ERR_INVALID_ARG;
    if (bits < 2 || bits > 4) return GPTQ_ERR_UNSUPPORTED;
    if (T == 0 || N == 0) return GPTQ_OK;
    if (!X || !packed || !scales || !zeros || !g_idx || !Y || G < 1 || ldx < K || ldy < N ||
        (flags & ~(GPTQ_DQ_RELU | GPTQ_DQ_BF16_OUT)))
        return GPTQ_ERR_INVALID_ARG;
    if (K % D_BK != 0 || K == 0 || ldx % 8 != 0 || (reinterpret_cast<uintptr_t>(X) & 15) ||
        (reinterpret_cast<uintptr_t>(g_idx) & 15) || T > (1ll << 31) - 1 || N > (1ll << 31) - 1)
        return GPTQ_ERR_UNSUPPORTED;
    auto enc = tma_encoder();
    if (!enc) return GPTQ_ERR_CUDA;
    CUtensorMap tx;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)T};
    cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
    cuuint32_t box[2] = {(cuuint32_t)D_BK, (cuuint32_t)D_BM};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return GPTQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DParams p;
    p.T = (int)T;
    p.N = (int)N;
    p.K = (int)K;
    p.tiles_n = (int)ceil_div(N, D_BN);
    p.ntiles = (int)(ceil_div(T, D_BM) * p.tiles_n);
    p.packed = packed;
    p.words = gptq_packed_words_per_row(K, bits);
    p.scales = scales;
    p.zeros = zeros;
    p.G = G;
    p.g_idx = g_idx;
    p.Y = Y;
    p.ldy = ldy;
    p.relu = (flags & GPTQ_DQ_RELU) ? 1 : 0;
    p.bf16_out = (flags & GPTQ_DQ_BF16_OUT) ? 1 : 0;
    // shared memory: stages + barriers, g_idx (int16), and the per-tile scale / zero tables
    // when they fit (otherwise the expansion reads scales and zeros from global memory)
    if (G > 32767 || K > 32768) return GPTQ_ERR_UNSUPPORTED;
    auto up16 = [](int64_t x) { return (x + 15) & ~int64_t(15); };
    p.g_off = D_RING + 256;
    p.sp = (int)(G | 1);
    int zq = (int)((G + 3) / 4);
    if ((zq & 1) == 0) ++zq;
    p.zp = 4 * zq;
    p.s_off = (int)up16(p.g_off + 2 * K);
    p.z_off = (int)up16(p.s_off + 4ll * D_BN * p.sp);
    const int64_t with_tab = p.z_off + (int64_t)D_BN * p.zp + 1024;
    p.tab = with_tab <= D_SMEM_MAX ? 1 : 0;
    const int smem = (int)(p.tab ? with_tab : up16(p.g_off + 2 * K) + 1024);
    if (smem > D_SMEM_MAX) return GPTQ_ERR_UNSUPPORTED;
    // Contiguous groups whose size is a multiple of the K step (no act_order) go to the exact
    // grouped kernel, the rest to the general one. Contiguity is checked on the device by
    // every CTA of both kernels (cta_groups_contiguous); both kernels are launched and the one
    // that does not apply returns at once.
    // (the grouped kernel has its own shared-memory layout: a copy of the parameters)
    const bool maybe_grouped = K % G == 0 && (K / G) % D_BK == 0;
    DParams pg = p;
    int gsmem = 0;
    if (maybe_grouped) {
        pg.gs = (int)(K / G);
        pg.s_off = (int)up16(D_RING + 256);
        pg.z_off = (int)up16(pg.s_off + 4ll * D_BN * G);
        const int64_t need = pg.z_off + (int64_t)D_BN * pg.zp + 1024;
        if (need <= D_SMEM_MAX) gsmem = (int)need;
    }
    const bool grouped = gsmem > 0;
    p.gs = grouped ? pg.gs : 0;   // the general kernel steps aside when the grouped one applies
    // the call's status word: static device memory, cleared on the stream (no allocation)
    int* status = nullptr;
    GPTQ_CUDA_TRY(call_status_word(s, &status));
    p.status = status;
    pg.status = status;
    const int grid = std::min(p.ntiles, device_sm_count());
    if (grouped) {
        auto gk = bits == 2 ? dequant_matmul_grouped_kernel<2>
                : bits == 3 ? dequant_matmul_grouped_kernel<3> : dequant_matmul_grouped_kernel<4>;
        GPTQ_CUDA_TRY(cudaFuncSetAttribute(gk, cudaFuncAttributeMaxDynamicSharedMemorySize, gsmem));
        GPTQ_LAUNCH(K_DEQUANT_MM, s, gk<<<grid, GQ_THREADS, gsmem, s>>>(tx, pg));
        GPTQ_LAUNCH_CHECK();
    }
    auto kern = p.tab ? (bits == 2 ? dequant_matmul_kernel<2, true> : bits == 3 ? dequant_matmul_kernel<3, true>
                                                                    : dequant_matmul_kernel<4, true>)
                      : (bits == 2 ? dequant_matmul_kernel<2, false> : bits == 3 ? dequant_matmul_kernel<3, false>
                                                                      : dequant_matmul_kernel<4, false>);
    GPTQ_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    GPTQ_LAUNCH(K_DEQUANT_MM, s, kern<<<grid, D_THREADS, smem, s>>>(tx, p));
    GPTQ_LAUNCH_CHECK();
    return finish_call(status, s);
}

namespace gptq {
// this file's copy of the pipeline-wait limit (the library's test hook sets every copy)
cudaError_t dequant_set_wait_limit(unsigned long long ns) { return set_pipeline_wait_limit_this_unit(ns); }
}  // namespace gptq
