// tc_gemm.cu — fp32-accurate NT GEMM on the 5th-generation tensor cores (3xTF32).
//
// C = beta * C + alpha * A * B^T for fp32 A (M x K) and B (N x K), both K-major. Each
// operand comes pre-split into hi (the fp32 value with its low 13 mantissa bits cleared,
// so exactly a TF32 number) and lo = value - hi (exact in fp32); the product is
// Ahi*Bhi + Ahi*Blo + Alo*Bhi, which leaves an error of order 2^-20 relative per term
// (the dropped Alo*Blo and the TF32 rounding of the lo parts), against 2^-11 for one TF32
// pass. Accumulation is fp32 in TMEM.
//
// Structure (one CTA per SM, persistent over 128 x BN output tiles). Variants:
//   BN = 128, 2-stage ring, the C tile in four chunk buffers (the default);
//   BN = 64, the same for a latency-critical launch too small to fill its SMs with
//     128-wide tiles;
//   deep (large launches with long K): C in two rotating chunk buffers, which frees the
//     shared memory for a third 64 KB stage (BN = 128) or for 128 x 256 tiles (two 96 KB
//     stages, when N >= 1024).
//   warp 0      TMA producer: per 32-wide K step, the four fp32 boxes Ahi, Alo (128 x 32)
//               and Bhi, Blo (BN x 32) (128-byte swizzle, K-major) into the ring
//   warp 1      single-thread tcgen05.mma issuer, kind::tf32, M = 128, N = BN, K = 8 per
//               instruction, three products per K step, into one of two TMEM
//               accumulators (BN columns each)
//   warps 2..5  epilogue: TMEM -> registers, combined with the C tile in shared memory
//               (brought by TMA: by the producer while the tile's MMAs run, or, in the
//               deep variant, by the epilogue's storer one chunk buffer ahead), stored
//               back by TMA in 32-column chunks; overlaps the MMAs of the next tile in the
//               other accumulator
// Every mbarrier wait is bounded (GPTQ_ERR_TIMEOUT into *status, then unwind).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc_gemm.cuh"

namespace gptq {

namespace {

// Output tiles are 128 rows x BN columns, BN = 128, or 64 for launches too small to fill
// their SMs with 128-wide tiles (twice the CTAs, each with half the MMAs and epilogue).
constexpr int G_BM = 128, G_BK = 32, G_THREADS = 192;
// K step of the 128 x 256 variant's operand ring (16: four 48 KB stages; 32: two 96 KB)
#ifndef GPTQ_GEMM_WIDE_KB
#define GPTQ_GEMM_WIDE_KB 16
#endif
constexpr int kWideKB = GPTQ_GEMM_WIDE_KB;
#ifndef GPTQ_GEMM_TM_INNER
#define GPTQ_GEMM_TM_INNER 1
#endif
constexpr int G_BOX = G_BM * G_BK * 4;         // 16 KB: one 128 x 32 fp32 box (a C chunk)
// KB: the K step of the operand ring in fp32 columns. 32 (128-byte rows, 128-byte swizzle);
// or 16 (64-byte rows, 64-byte swizzle), which halves a stage so twice as many stages fit
// in the same shared memory and a stage's load has more K steps of MMAs to hide behind.
template <int BN, bool DEEP = false, int KB = G_BK>
struct GTile {
    static constexpr int ABOX = G_BM * KB * 4;                      // one 128 x KB fp32 box of A
    static constexpr int BBOX = BN * KB * 4;                        // one BN x KB fp32 box of B
    static constexpr int STAGE = 2 * ABOX + 2 * BBOX;               // Ahi, Alo, Bhi, Blo
    // ring depth: 3 for the deep 128-wide variant (large launches with long K: a stage
    // arrives ~1.1-1.2k cycles after its TMA issue under full load, more than one K step of
    // MMAs), whose C tile then streams through two rotating 32-column chunk buffers; 4 for
    // the deep 256-wide variant with 16-wide K steps; else 2
    static constexpr int STAGES = (DEEP && BN == 128 && KB == 32) ? 3 : (DEEP && KB == 16) ? 4 : 2;
    static constexpr int CB = DEEP ? 2 : BN / 32;                   // C chunk buffers
    static constexpr int NCH = BN / 32;                             // 32-column C chunks
    static constexpr int CBUF = CB * G_BOX;                         // C chunk buffers
    static constexpr int SMEM = STAGES * STAGE + CBUF + 1024 + 256;
    static constexpr uint32_t TMEM_COLS = 2 * BN;                   // two accumulators
    // operand layout: 8-row core-matrix groups KB * 4 * 8 bytes apart; swizzle mode of the
    // shared-memory descriptor (2 = 128-byte, 4 = 64-byte)
    static constexpr uint32_t SBO = KB * 4 * 8;
    static constexpr uint64_t SWZ = KB == 32 ? 2 : 4;
    // kind::tf32: D fp32 (bits 4-5 = 1), A/B TF32 (2), both K-major, N >> 3, M >> 4
    static constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                      ((uint32_t)(G_BM >> 4) << 24);
};

static_assert(GTile<64>::SMEM <= 232448 && GTile<128>::SMEM <= 232448 && GTile<128, true>::SMEM <= 232448 &&
                  GTile<256, true>::SMEM <= 232448 && GTile<256, true, 16>::SMEM <= 232448,
              "shared memory per CTA");
static_assert(2 * GTile<256, true, 16>::STAGES + 12 < 30, "barrier slots");

struct GParams {
    int M, N, K;
    float alpha, beta;
    int tiles_m, tiles_n, ntiles, lower_only;
    int tm_inner;   // full launches: tile rows vary fastest (a wave spans all of A)
    int bn;     // tile width in columns
    int* status;
    // optional TF32 split of the result: mode 1 hi[r][c], mode 2 (transposed) hi[c][r]
    float* ohi;
    float* olo;
    int64_t old_;
    int omode;
    int orow0;
    int ovec;   // row-major split rows are 16-byte aligned
};

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// barrier over the 128 epilogue threads that also ANDs a predicate across them, so that
// all epilogue warps take the same branch after a bounded wait
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "barrier.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)(v ? 1 : 0))
        : "memory");
    return r != 0;
}

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            set_status(status, GPTQ_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// tiles of tile row r that reach the diagonal or below it (lower_only)
__host__ __device__ __forceinline__ int lower_tiles_in_row(int r, int bn, int tiles_n) {
    const int c = (r * G_BM + G_BM - 1) / bn + 1;
    return c < tiles_n ? c : tiles_n;
}

// linear tile index -> (tm, tn); with lower_only the tiles that reach the diagonal or
// below it, row by row
__device__ __forceinline__ void tile_of(const GParams& p, int t, int& tm, int& tn) {
    if (!p.lower_only) {
        if (p.tm_inner) {
            tm = t % p.tiles_m;
            tn = t / p.tiles_m;
        } else {
            tm = t / p.tiles_n;
            tn = t % p.tiles_n;
        }
        return;
    }
    int r = 0;
    for (;;) {
        const int c = lower_tiles_in_row(r, p.bn, p.tiles_n);
        if (t < c) break;
        t -= c;
        ++r;
    }
    tm = r;
    tn = t;
}

// The C tile moves through shared memory by TMA in both directions: the producer loads it
// (when beta != 0) while the MMAs of the tile run, the epilogue combines it with the
// accumulator in place and stores it back with TMA, so no thread waits on a global load.
template <int BN, bool DEEP, int KB = G_BK>
__global__ void __launch_bounds__(G_THREADS, 1) tc_gemm_nt_kernel(const __grid_constant__ CUtensorMap tAh,
                                                                  const __grid_constant__ CUtensorMap tAl,
                                                                  const __grid_constant__ CUtensorMap tBh,
                                                                  const __grid_constant__ CUtensorMap tBl,
                                                                  const __grid_constant__ CUtensorMap tC,
                                                                  const GParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using T = GTile<BN, DEEP, KB>;
    constexpr int G_STAGES = T::STAGES;
    uint8_t* cbuf = smem + G_STAGES * T::STAGE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(cbuf + T::CBUF);
    // barriers occupy slots 0 .. 2 * STAGES + 12 (at most 20) of the 32 in the 256-byte area
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 30);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 31);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(smem), cbase = smem_u32(cbuf), bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (G_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * G_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * G_STAGES + 2 + b); };
    // the C tile moves as four 32-column chunks, each with its own full / empty barrier,
    // so the next tile's chunk c loads as soon as this tile's chunk c has been stored
    auto cfull_bar = [&](int c) { return bar0 + 8u * (2 * G_STAGES + 4 + c); };
    auto cempty_bar = [&](int c) { return bar0 + 8u * (2 * G_STAGES + 8 + c); };
    const uint32_t drain_bar = bar0 + 8u * (2 * G_STAGES + 12);
    const bool load_c = p.beta != 0.0f;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4);
        }
        for (int c = 0; c < T::CB; ++c) {
            mbar_init(cfull_bar(c), 1);
            mbar_init(cempty_bar(c), 1);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tAh);
        tma_prefetch_desc(&tAl);
        tma_prefetch_desc(&tBh);
        tma_prefetch_desc(&tBl);
        tma_prefetch_desc(&tC);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int ktiles = (p.K + KB - 1) / KB;
    pdl_wait();      // operands and C may be the previous kernel's output
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------- TMA producer -------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_par = 0, cph = 0, c_issued = 0, c_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
                int tm, tn;
                tile_of(p, t, tm, tn);
                for (int kt = 0; kt < ktiles; ++kt) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full_bar(stage), T::STAGE);
                    const uint32_t sa = sbase + stage * T::STAGE;
                    const int x = kt * KB;
                    tma_load_2d(sa, &tAh, full_bar(stage), x, tm * G_BM);
                    tma_load_2d(sa + T::ABOX, &tAl, full_bar(stage), x, tm * G_BM);
                    tma_load_2d(sa + 2 * T::ABOX, &tBh, full_bar(stage), x, tn * BN);
                    tma_load_2d(sa + 2 * T::ABOX + T::BBOX, &tBl, full_bar(stage), x, tn * BN);
                    issued |= 1u << stage;
                    issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (load_c && !DEEP) {
                    // chunk c of the C buffer is free once the previous tile's store of it
                    // has been read
                    for (int c = 0; c < T::NCH && ok; ++c) {
                        if (!mbar_wait(cempty_bar(c), cph ^ 1u, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(cfull_bar(c), G_BOX);
                        tma_load_2d(cbase + c * G_BOX, &tC, cfull_bar(c), tn * BN + 32 * c, tm * G_BM);
                        c_issued |= 1u << c;
                        c_par = (c_par & ~(1u << c)) | (cph << c);
                    }
                    if (!ok) break;
                    cph ^= 1u;
                }
            }
            for (int s = 0; s < G_STAGES; ++s)
                if (issued & (1u << s)) drain_wait(full_bar(s), (issued_par >> s) & 1u, p.status);
            for (int c = 0; c < (DEEP ? 0 : T::NCH); ++c)
                if (c_issued & (1u << c)) drain_wait(cfull_bar(c), (c_par >> c) & 1u, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer ---------------------------------
        if (lane == 0) {
            int stage = 0, abuf = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
                if (!mbar_wait(tempty_bar(abuf), aphase ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t dt = tmem_base + (uint32_t)(abuf * BN);
                for (int kt = 0; kt < ktiles; ++kt) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + stage * T::STAGE;
#pragma unroll
                    for (int kk = 0; kk < KB / 8; ++kk) {
                        // 8 TF32 = 32 bytes along K inside the swizzled row
                        const uint32_t off = kk * 32;
                        const uint64_t ah = smem_desc(sa + off, 16, T::SBO, T::SWZ);
                        const uint64_t al = smem_desc(sa + T::ABOX + off, 16, T::SBO, T::SWZ);
                        const uint64_t bh = smem_desc(sa + 2 * T::ABOX + off, 16, T::SBO, T::SWZ);
                        const uint64_t bl = smem_desc(sa + 2 * T::ABOX + T::BBOX + off, 16, T::SBO, T::SWZ);
                        umma_tf32(dt, ah, bh, T::IDESC, (kt > 0 || kk > 0) ? 1u : 0u);
                        umma_tf32(dt, ah, bl, T::IDESC, 1u);
                        umma_tf32(dt, al, bh, T::IDESC, 1u);
                    }
                    umma_commit(empty_bar(stage));
                    if (++stage == G_STAGES) {
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
            umma_commit(drain_bar);
            drain_wait(drain_bar, 0, p.status);
        }
    } else if constexpr (DEEP) {
        // ------------- epilogue (4 warps), C through two rotating chunk buffers ------------
        // The storer keeps each buffer filled one use ahead: chunks 0 and 1 of the CTA's first
        // tile at the start; chunk c + 2, or chunk c - 2 of the CTA's next tile, as soon as
        // the store of chunk c has read the buffer (a TMA load of C, or without C just an
        // arrive). Every thread waits for a buffer's fill before using it.
        const int q = warp & 3;
        const int rl = 32 * q + lane;            // row of the tile this thread owns
        const bool storer = (threadIdx.x == 64);
        int abuf = 0;
        uint32_t aphase = 0, cph = 0;            // cph bit b: phase of buffer b's next fill
        uint32_t issued0 = 0, issued1 = 0, consumed0 = 0, consumed1 = 0;   // per buffer
        auto fill = [&](int b, int ftm, int ftn, int c) {
            if (load_c) {
                mbar_expect_tx(cfull_bar(b), G_BOX);
                tma_load_2d(cbase + b * G_BOX, &tC, cfull_bar(b), ftn * BN + 32 * c, ftm * G_BM);
            } else {
                mbar_arrive(cfull_bar(b));
            }
            if (b) ++issued1; else ++issued0;
        };
        if (storer && (int)blockIdx.x < p.ntiles) {
            int tm0, tn0;
            tile_of(p, blockIdx.x, tm0, tn0);
            fill(0, tm0, tn0, 0);
            fill(1, tm0, tn0, 1);
        }
        bool alive = true;
        for (int t = blockIdx.x; t < p.ntiles && alive; t += gridDim.x) {
            int tm, tn, ntm = 0, ntn = 0;
            tile_of(p, t, tm, tn);
            const bool has_next = t + (int)gridDim.x < p.ntiles;
            if (has_next) tile_of(p, t + (int)gridDim.x, ntm, ntn);
            if (!epi_all(mbar_wait(tfull_bar(abuf), aphase, abort_flag, p.status))) break;
            tc_fence_after();
            const int row = tm * G_BM + rl;
            const uint32_t ta = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(abuf * BN);
#pragma unroll 1
            for (int c = 0; c < T::NCH; ++c) {
                const int b = c & 1;
                if (!epi_all(mbar_wait(cfull_bar(b), (cph >> b) & 1u, abort_flag, p.status))) {
                    alive = false;
                    break;
                }
                cph ^= 1u << b;
                if (b) ++consumed1; else ++consumed0;
                uint32_t v[32];
                tmem_ld_32x32b_x32(ta + 32 * c, v);
                tmem_ld_wait();
                uint8_t* brow = cbuf + b * G_BOX + rl * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4* ptr = reinterpret_cast<float4*>(brow + ((j ^ (rl & 7)) << 4));
                    float4 o = make_float4(p.alpha * __uint_as_float(v[4 * j]), p.alpha * __uint_as_float(v[4 * j + 1]),
                                           p.alpha * __uint_as_float(v[4 * j + 2]),
                                           p.alpha * __uint_as_float(v[4 * j + 3]));
                    if (load_c) {
                        const float4 cv = *ptr;
                        o.x = fmaf(p.beta, cv.x, o.x);
                        o.y = fmaf(p.beta, cv.y, o.y);
                        o.z = fmaf(p.beta, cv.z, o.z);
                        o.w = fmaf(p.beta, cv.w, o.w);
                    }
                    *ptr = o;
                    const int gc0 = tn * BN + 32 * c + 4 * j;
                    if (p.omode == 1 && row < p.M && row >= p.orow0 && gc0 + 3 < p.N && p.ovec) {
                        // row-major split, four columns at once (16-byte stores)
                        float4 h4;
                        h4.x = __uint_as_float(__float_as_uint(o.x) & 0xFFFFE000u);
                        h4.y = __uint_as_float(__float_as_uint(o.y) & 0xFFFFE000u);
                        h4.z = __uint_as_float(__float_as_uint(o.z) & 0xFFFFE000u);
                        h4.w = __uint_as_float(__float_as_uint(o.w) & 0xFFFFE000u);
                        const int64_t at = (int64_t)(row - p.orow0) * p.old_ + gc0;
                        *reinterpret_cast<float4*>(p.ohi + at) = h4;
                        *reinterpret_cast<float4*>(p.olo + at) = make_float4(o.x - h4.x, o.y - h4.y, o.z - h4.z, o.w - h4.w);
                    } else if (p.omode && row < p.M && row >= p.orow0) {
                        const float o4[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int gc = tn * BN + 32 * c + 4 * j + e;
                            if (gc < p.N) {
                                const float h = __uint_as_float(__float_as_uint(o4[e]) & 0xFFFFE000u);
                                const int64_t orow = row - p.orow0;
                                const int64_t at = (p.omode == 1) ? orow * p.old_ + gc : (int64_t)gc * p.old_ + orow;
                                p.ohi[at] = h;
                                p.olo[at] = o4[e] - h;
                            }
                        }
                    }
                }
                fence_proxy_async_smem();   // make the chunk visible to TMA
                epi_barrier();
                if (storer) {
                    tma_store_2d(&tC, cbase + b * G_BOX, tn * BN + 32 * c, tm * G_BM);
                    bulk_commit();
                    bulk_wait_read0();       // the store has read buffer b: refill it
                    if (c + 2 < T::NCH)
                        fill(b, tm, tn, c + 2);
                    else if (has_next)
                        fill(b, ntm, ntn, c + 2 - T::NCH);
                }
            }
            if (!alive) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(abuf));   // the accumulator is free again
            if (++abuf == 2) {
                abuf = 0;
                aphase ^= 1u;
            }
        }
        if (storer) {
            bulk_wait0();
            // a fill issued but never waited for (an aborted tile): let its copy land first
            if (issued0 > consumed0) drain_wait(cfull_bar(0), (issued0 - 1u) & 1u, p.status);
            if (issued1 > consumed1) drain_wait(cfull_bar(1), (issued1 - 1u) & 1u, p.status);
        }
    } else {
        // ------------------------------- epilogue (4 warps) -------------------------
        const int q = warp & 3;
        const int rl = 32 * q + lane;            // row of the tile this thread owns
        const bool storer = (threadIdx.x == 64);
        int abuf = 0;
        uint32_t aphase = 0, cph = 0;
        bool alive = true;
        for (int t = blockIdx.x; t < p.ntiles && alive; t += gridDim.x) {
            int tm, tn;
            tile_of(p, t, tm, tn);
            if (!epi_all(mbar_wait(tfull_bar(abuf), aphase, abort_flag, p.status))) break;
            tc_fence_after();
            const int row = tm * G_BM + rl;
            const uint32_t ta = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(abuf * BN);
#pragma unroll 1
            for (int c = 0; c < T::NCH; ++c) {
                if (load_c && !epi_all(mbar_wait(cfull_bar(c), cph, abort_flag, p.status))) {
                    alive = false;
                    break;
                }
                uint32_t v[32];
                tmem_ld_32x32b_x32(ta + 32 * c, v);
                tmem_ld_wait();
                uint8_t* brow = cbuf + c * G_BOX + rl * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4* ptr = reinterpret_cast<float4*>(brow + ((j ^ (rl & 7)) << 4));
                    float4 o = make_float4(p.alpha * __uint_as_float(v[4 * j]), p.alpha * __uint_as_float(v[4 * j + 1]),
                                           p.alpha * __uint_as_float(v[4 * j + 2]),
                                           p.alpha * __uint_as_float(v[4 * j + 3]));
                    if (load_c) {
                        const float4 cv = *ptr;
                        o.x = fmaf(p.beta, cv.x, o.x);
                        o.y = fmaf(p.beta, cv.y, o.y);
                        o.z = fmaf(p.beta, cv.z, o.z);
                        o.w = fmaf(p.beta, cv.w, o.w);
                    }
                    *ptr = o;
                    const int gc0 = tn * BN + 32 * c + 4 * j;
                    if (p.omode == 1 && row < p.M && row >= p.orow0 && gc0 + 3 < p.N && p.ovec) {
                        // row-major split, four columns at once (16-byte stores)
                        float4 h4;
                        h4.x = __uint_as_float(__float_as_uint(o.x) & 0xFFFFE000u);
                        h4.y = __uint_as_float(__float_as_uint(o.y) & 0xFFFFE000u);
                        h4.z = __uint_as_float(__float_as_uint(o.z) & 0xFFFFE000u);
                        h4.w = __uint_as_float(__float_as_uint(o.w) & 0xFFFFE000u);
                        const int64_t at = (int64_t)(row - p.orow0) * p.old_ + gc0;
                        *reinterpret_cast<float4*>(p.ohi + at) = h4;
                        *reinterpret_cast<float4*>(p.olo + at) = make_float4(o.x - h4.x, o.y - h4.y, o.z - h4.z, o.w - h4.w);
                    } else if (p.omode && row < p.M && row >= p.orow0) {
                        const float o4[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int gc = tn * BN + 32 * c + 4 * j + e;
                            if (gc < p.N) {
                                const float h = __uint_as_float(__float_as_uint(o4[e]) & 0xFFFFE000u);
                                const int64_t orow = row - p.orow0;
                                const int64_t at = (p.omode == 1) ? orow * p.old_ + gc : (int64_t)gc * p.old_ + orow;
                                p.ohi[at] = h;
                                p.olo[at] = o4[e] - h;
                            }
                        }
                    }
                }
                fence_proxy_async_smem();   // make the chunk visible to TMA
                epi_barrier();
                if (storer) {
                    // store chunk c; once the store of chunk c-1 has read its buffer, the
                    // producer may load the next tile's chunk c-1 there. (Writes of the next
                    // tile's chunk c-1 by the other threads come after a later barrier.)
                    tma_store_2d(&tC, cbase + c * G_BOX, tn * BN + 32 * c, tm * G_BM);
                    bulk_commit();
                    if (c > 0) {
                        bulk_wait_read1();
                        if (load_c) mbar_arrive(cempty_bar(c - 1));
                    }
                }
            }
            if (!alive) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(abuf));   // the accumulator is free again
            if (storer) {
                bulk_wait_read0();
                if (load_c) mbar_arrive(cempty_bar(T::NCH - 1));
            }
            if (++abuf == 2) {
                abuf = 0;
                aphase ^= 1u;
            }
            if (load_c) cph ^= 1u;
        }
        if (storer) bulk_wait0();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, T::TMEM_COLS);
    }
}

__device__ __forceinline__ void split1(float a, float& hi, float& lo) {
    hi = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
    lo = a - hi;
}

__global__ void split_rows_kernel(const float* __restrict__ A, int64_t lda, int rows, int K, float* __restrict__ hi,
                                  float* __restrict__ lo, int ldk) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.y;
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < K; k += gridDim.x * blockDim.x) {
        float h, l;
        split1(A[(int64_t)r * lda + k], h, l);
        hi[(int64_t)r * ldk + k] = h;
        lo[(int64_t)r * ldk + k] = l;
    }
}

// the same with one float4 per thread (K, lda, ldk multiples of 4, 16-byte aligned rows)
__global__ void __launch_bounds__(256) split_rows4_kernel(const float* __restrict__ A, int64_t lda, int rows, int K,
                                                         float* __restrict__ hi, float* __restrict__ lo, int ldk) {
    pdl_wait();
    pdl_trigger();
    const int k4 = K >> 2;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)rows * k4) return;
    const int64_t r = idx / k4;
    const int k = (int)(idx - r * k4) * 4;
    const float4 v = *reinterpret_cast<const float4*>(A + r * lda + k);
    float4 h, l;
    split1(v.x, h.x, l.x);
    split1(v.y, h.y, l.y);
    split1(v.z, h.z, l.z);
    split1(v.w, h.w, l.w);
    *reinterpret_cast<float4*>(hi + r * ldk + k) = h;
    *reinterpret_cast<float4*>(lo + r * ldk + k) = l;
}

// B (K x N block, row stride ld) -> hi/lo (N x ldk), transposed through a 32 x 33 tile
__global__ void __launch_bounds__(256) split_cols_kernel(const float* __restrict__ B, int64_t ld, int K, int N,
                                                        float* __restrict__ hi, float* __restrict__ lo, int ldk) {
    __shared__ float tile[32][33];
    pdl_wait();
    pdl_trigger();
    const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8) {
        const int k = k0 + r, n = n0 + tx;
        tile[r][tx] = (k < K && n < N) ? B[(int64_t)k * ld + n] : 0.0f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int n = n0 + r, k = k0 + tx;
        if (n < N && k < K) {
            float h, l;
            split1(tile[tx][r], h, l);
            hi[(int64_t)n * ldk + k] = h;
            lo[(int64_t)n * ldk + k] = l;
        }
    }
}

// The same with 16-byte accesses on both sides (N, ld and ldk multiples of 4, 16-byte
// aligned bases): a 64 x 64 tile per CTA, read as rows of B, written as rows of hi/lo.
constexpr int SC_T = 64;
__global__ void __launch_bounds__(256) split_cols4_kernel(const float* __restrict__ B, int64_t ld, int K, int N,
                                                         float* __restrict__ hi, float* __restrict__ lo, int ldk,
                                                         int strict_lower) {
    __shared__ float tile[SC_T][SC_T + 1];
    pdl_wait();
    pdl_trigger();
    const int k0 = blockIdx.y * SC_T, n0 = blockIdx.x * SC_T;
    if (strict_lower && n0 + SC_T <= k0) return;   // every output n < k: never read
    const int c4 = (threadIdx.x & 15) * 4, r = threadIdx.x >> 4;   // 16 float4 per row, 16 rows per pass
#pragma unroll
    for (int rr = 0; rr < SC_T; rr += 16) {
        const int k = k0 + rr + r, n = n0 + c4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (k < K && n < N) v = *reinterpret_cast<const float4*>(B + (int64_t)k * ld + n);   // N % 4 == 0
        tile[rr + r][c4] = v.x;
        tile[rr + r][c4 + 1] = v.y;
        tile[rr + r][c4 + 2] = v.z;
        tile[rr + r][c4 + 3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < SC_T; rr += 16) {
        const int n = n0 + rr + r, k = k0 + c4;
        if (n >= N || k >= K) continue;
        float4 h, l;
        split1(tile[c4][rr + r], h.x, l.x);
        split1(tile[c4 + 1][rr + r], h.y, l.y);
        split1(tile[c4 + 2][rr + r], h.z, l.z);
        split1(tile[c4 + 3][rr + r], h.w, l.w);
        float* ph = hi + (int64_t)n * ldk + k;
        float* pl = lo + (int64_t)n * ldk + k;
        if (k + 3 < K) {
            *reinterpret_cast<float4*>(ph) = h;
            *reinterpret_cast<float4*>(pl) = l;
        } else {
            const float hs[4] = {h.x, h.y, h.z, h.w}, ls[4] = {l.x, l.y, l.z, l.w};
            for (int e = 0; e < 4 && k + e < K; ++e) {
                ph[e] = hs[e];
                pl[e] = ls[e];
            }
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() { return tma_encoder(); }

// box of box_rows rows x kb fp32 columns: kb = 32 (128-byte swizzle) or 16 (64-byte swizzle)
bool make_map(CUtensorMap* m, const float* base, int rows, int K, int64_t ldk, int box_rows = G_BM, int kb = G_BK) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ldk * 4};
    cuuint32_t box[2] = {(cuuint32_t)kb, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, kb == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
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

cudaError_t split_rows(int id, const float* A, int64_t lda, int rows, int K, float* hi, float* lo, int ldk,
                       cudaStream_t s, bool pdl) {
    if (rows <= 0 || K <= 0) return cudaSuccess;
    dim3 grid((unsigned)std::min((K + 255) / 256, 8), (unsigned)rows);
    const bool vec = (K % 4 == 0) && (lda % 4 == 0) && (ldk % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(hi) |
                       reinterpret_cast<uintptr_t>(lo)) % 16 == 0);
    cudaError_t e = cudaSuccess;
    if (vec) {
        const unsigned blocks = (unsigned)(((int64_t)rows * (K / 4) + 255) / 256);
        if (pdl)
            GPTQ_LAUNCH(id, s, e = launch_pdl(split_rows4_kernel, dim3(blocks), dim3(256), 0, s, A, lda, rows, K, hi, lo, ldk));
        else
            GPTQ_LAUNCH(id, s, split_rows4_kernel<<<blocks, 256, 0, s>>>(A, lda, rows, K, hi, lo, ldk));
    } else if (pdl) {
        GPTQ_LAUNCH(id, s, e = launch_pdl(split_rows_kernel, grid, dim3(256), 0, s, A, lda, rows, K, hi, lo, ldk));
    } else {
        GPTQ_LAUNCH(id, s, split_rows_kernel<<<grid, 256, 0, s>>>(A, lda, rows, K, hi, lo, ldk));
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t split_cols(int id, const float* B, int64_t ld, int K, int N, float* hi, float* lo, int ldk,
                       cudaStream_t s, bool pdl, bool strict_lower) {
    if (K <= 0 || N <= 0) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    const bool vec = (N % 4 == 0) && (ld % 4 == 0) && (ldk % 4 == 0) &&
                     ((reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(hi) |
                       reinterpret_cast<uintptr_t>(lo)) % 16 == 0);
    if (vec) {
        dim3 grid((unsigned)((N + SC_T - 1) / SC_T), (unsigned)((K + SC_T - 1) / SC_T));
        if (pdl)
            GPTQ_LAUNCH(id, s, e = launch_pdl(split_cols4_kernel, grid, dim3(256), 0, s, B, ld, K, N, hi, lo, ldk,
                                              (int)strict_lower));
        else
            GPTQ_LAUNCH(id, s, split_cols4_kernel<<<grid, 256, 0, s>>>(B, ld, K, N, hi, lo, ldk, (int)strict_lower));
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    dim3 grid((unsigned)((N + 31) / 32), (unsigned)((K + 31) / 32));
    if (pdl)
        GPTQ_LAUNCH(id, s, e = launch_pdl(split_cols_kernel, grid, dim3(256), 0, s, B, ld, K, N, hi, lo, ldk));
    else
        GPTQ_LAUNCH(id, s, split_cols_kernel<<<grid, 256, 0, s>>>(B, ld, K, N, hi, lo, ldk));
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

bool tc_gemm_nt_ok(const float* C, int64_t ldc) {
    return (reinterpret_cast<uintptr_t>(C) % 16 == 0) && (ldc % 4 == 0) && encoder() != nullptr;
}

cudaError_t tc_gemm_nt(int id, int M, int N, int K, float alpha, const float* Ahi, const float* Alo, const float* Bhi,
                       const float* Blo, int ldk, float beta, float* C, int64_t ldc, bool lower_only, int* status,
                       cudaStream_t s, GemmOpts out) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (out.ldb == 0) out.ldb = ldk;
    static const int sms = device_sm_count();
    const int cap = out.max_ctas > 0 ? std::min(out.max_ctas, sms) : sms;
    auto count_tiles = [&](int bn, int& tiles_n) {
        const int tiles_m = (M + G_BM - 1) / G_BM;
        tiles_n = (N + bn - 1) / bn;
        if (!lower_only) return tiles_m * tiles_n;
        int cnt = 0;
        for (int r = 0; r < tiles_m; ++r) cnt += lower_tiles_in_row(r, bn, tiles_n);
        return cnt;
    };
    // 64-column tiles for a latency-critical launch whose 64-wide tiles still fit in one
    // wave of its CTAs: twice the CTAs, each with half the epilogue (the per-CTA MMA time
    // stays: a tcgen05.mma with N = 64 takes about as long as one with N = 128)
    int tn128 = 0, tn64 = 0;
    const int nt128 = count_tiles(128, tn128), nt64 = count_tiles(64, tn64);
    const int bn = (out.narrow_ok && nt128 < cap && nt64 <= cap) ? 64 : 128;
    // the deep variant for large launches: at least two waves of tiles, K of 8 steps or
    // more; 128 x 256 tiles (two 96 KB stages: each K step's MMAs take twice as long, which
    // covers a stage's load, and a quarter less operand traffic per flop) when N is large
    int tn256 = 0;
    const int nt256 = count_tiles(256, tn256);
    const bool deep = bn == 128 && nt128 >= 2 * cap && K >= 8 * G_BK;
    const bool wide = deep && N >= 1024 && nt256 >= cap;
    const int tw = wide ? 256 : bn;   // the launch's tile width
    const int kb = wide ? kWideKB : G_BK;   // the operand ring's K step
    CUtensorMap tah, tal, tbh, tbl, tcm;
    if (!make_map(&tah, Ahi, M, K, ldk, G_BM, kb) || !make_map(&tal, Alo, M, K, ldk, G_BM, kb) ||
        !make_map(&tbh, Bhi, N, K, out.ldb, tw, kb) || !make_map(&tbl, Blo, N, K, out.ldb, tw, kb) ||
        !make_map(&tcm, C, M, N, ldc))
        return cudaErrorInvalidValue;
    GParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.bn = tw;
    p.tiles_m = (M + G_BM - 1) / G_BM;
    p.tiles_n = tw == 64 ? tn64 : tw == 256 ? tn256 : tn128;
    p.lower_only = lower_only ? 1 : 0;
    p.ntiles = tw == 64 ? nt64 : tw == 256 ? nt256 : nt128;
    // The tiles a wave of CTAs runs together read all of the operand they span in the
    // other direction: by rows, all of B (N x K) per wave; with tile rows innermost, all of
    // A (M x K). The one read again wave after wave should be the smaller.
    p.tm_inner = (!lower_only && M < N) ? GPTQ_GEMM_TM_INNER : 0;
    p.status = status;
    p.ohi = out.hi;
    p.olo = out.lo;
    p.old_ = out.ld;
    p.omode = out.hi ? out.mode : 0;
    p.orow0 = (int)out.row0;
    p.ovec = (out.hi && (out.ld % 4 == 0) &&
              ((reinterpret_cast<uintptr_t>(out.hi) | reinterpret_cast<uintptr_t>(out.lo)) % 16 == 0)) ? 1 : 0;
    if (p.ntiles == 0) return cudaSuccess;
    const int grid = std::min(p.ntiles, cap);
    auto kern = bn == 64 ? tc_gemm_nt_kernel<64, false>
              : wide    ? (kWideKB == 16 ? tc_gemm_nt_kernel<256, true, 16> : tc_gemm_nt_kernel<256, true, 32>)
              : deep    ? tc_gemm_nt_kernel<128, true>
                        : tc_gemm_nt_kernel<128, false>;
    const int smem = bn == 64 ? GTile<64>::SMEM
                   : wide    ? (kWideKB == 16 ? GTile<256, true, 16>::SMEM : GTile<256, true, 32>::SMEM)
                   : deep    ? GTile<128, true>::SMEM
                             : GTile<128>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (out.pdl) {
        GPTQ_LAUNCH(id, s, e = launch_pdl(kern, dim3(grid), dim3(G_THREADS), (size_t)smem, s, tah, tal, tbh, tbl, tcm,
                                          p));
        if (e != cudaSuccess) return e;
    } else {
        GPTQ_LAUNCH(id, s, kern<<<grid, G_THREADS, smem, s>>>(tah, tal, tbh, tbl, tcm, p));
    }
    return cudaGetLastError();
}

}  // namespace gptq

namespace gptq {
// this file's copy of the pipeline-wait limit (the library's test hook sets every copy)
cudaError_t tc_gemm_set_wait_limit(unsigned long long ns) { return set_pipeline_wait_limit_this_unit(ns); }
}  // namespace gptq
