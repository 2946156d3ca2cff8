// quantize.cu — GPTQ's fixed-order column loop, round-to-nearest, g_idx and packing.
//
// The column loop (GPTQ's error-compensation loop page, its four steps; GPTQ guide page,
// "Source code", `gptq`) is run in 128-column blocks, the lazy-batch structure the guide
// page's "Simplifications" paragraph names (same result, block updates):
//
//   for each block [j0, j0+128):
//     gptq_block_kernel    rows in parallel (4 threads per row, 32 columns each in
//                          registers); U[blk, blk] in shared memory; for every column j:
//                          broadcast w_j inside the row's 4 lanes, q = grid(w_j),
//                          err = (w_j - q) / U[j][j], w_c -= err * U[j][c] for the block's
//                          columns (U is zero below the diagonal, so columns already done
//                          are untouched); group scales/zero points at each group start
//                          from the updated weights; Err[:, blk] kept for the update below
//     trailing update      W[:, j0+128:] -= Err * U[blk, j0+128:]   (fp32 GEMM)
//
// On the tensor-core path the trailing update is applied in two levels: blocks are grouped
// four at a time into super-blocks; after a block only the rest of its super-block is
// updated, and at the end of a super-block the columns past it are updated with the
// errors of all four blocks in one K = 512 product. The sum is the same (each column
// still receives every earlier block's correction before its own block runs); the large
// trailing matrix is read and written a quarter as often.
//
// The working copy of W lives in the caller's workspace, permuted into loop order with
// dead columns zeroed (guide page, "Source code": W[:, dead] = 0, W = W[:, perm]).
// Outputs go straight to the original column order.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "quant.cuh"
#include "sgemm.cuh"
#include "tc_gemm.cuh"

namespace gptq {

namespace {

constexpr int QB = 128;  // column block width
// Blocks per super-block of the deferred trailing update: inside a super-block only its
// own columns are updated after each block (K = 128); at its end everything past it, with
// K = sb * 128. Wide weights take 8 (fewer passes over their long trailing matrix), the
// others 4 (measured: 4096 x 14336 6.81 -> 6.60 ms with 8; 28672 x 4096 4.40 -> 4.54 ms).
#ifndef GPTQ_QUANT_SB_WIDE
#define GPTQ_QUANT_SB_WIDE 8
#endif
inline int super_blocks(int64_t cols) { return cols >= 8192 ? GPTQ_QUANT_SB_WIDE : 4; }

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct QuantWs {
    float* W;       // rows x cols working copy (loop order)
    float* Err;     // rows x QB
    float* ehi;     // rows x sb*QB: TF32 split of Err for the blocks of one super-block
    float* elo;
    float* uhi;     // cols x cols: TF32 split of U^T
    float* ulo;
    float* cur_s;   // rows: current scale (per-row grid, or a group wider than a block)
    float* cur_z;   // rows
    float* loss;    // rows
    int* status;
    size_t bytes;
};

QuantWs carve(void* base, int64_t rows, int64_t cols) {
    QuantWs w{};
    char* p = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* q = p + off;
        off = align256(off + bytes);
        return q;
    };
    w.W = reinterpret_cast<float*>(take(sizeof(float) * rows * cols));
    w.Err = reinterpret_cast<float*>(take(sizeof(float) * rows * QB));
    const int64_t sb = super_blocks(cols);
    w.ehi = reinterpret_cast<float*>(take(sizeof(float) * rows * sb * QB));
    w.elo = reinterpret_cast<float*>(take(sizeof(float) * rows * sb * QB));
    w.uhi = reinterpret_cast<float*>(take(sizeof(float) * cols * cols));
    w.ulo = reinterpret_cast<float*>(take(sizeof(float) * cols * cols));
    w.cur_s = reinterpret_cast<float*>(take(sizeof(float) * rows));
    w.cur_z = reinterpret_cast<float*>(take(sizeof(float) * rows));
    w.loss = reinterpret_cast<float*>(take(sizeof(float) * rows));
    w.status = reinterpret_cast<int*>(take(sizeof(int) * 4));
    w.bytes = off;
    return w;
}

bool group_ok(int group) { return group == 0 || (group > 0 && (group % QB == 0 || QB % group == 0)); }

// Wk[r][k] = dead[perm[k]] ? 0 : W[r][perm[k]]
// Four consecutive loop columns per thread (one 16-byte store when cols % 4 == 0), IW_ROWS
// rows per CTA so the permutation and dead flags are read once for several rows. A weight
// that is not finite (outside a dead column, which is never read) records
// GPTQ_ERR_NONFINITE.
constexpr int IW_ROWS = 4;
__global__ void __launch_bounds__(256) init_work_kernel(const float* __restrict__ W, int64_t rows, int64_t cols,
                                                        const int32_t* __restrict__ perm,
                                                        const uint8_t* __restrict__ dead, float* __restrict__ Wk,
                                                        int* __restrict__ status) {
    const int64_t k0 = 4 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
    if (k0 >= cols) return;
    const int nk = cols - k0 < 4 ? (int)(cols - k0) : 4;
    int64_t c[4];
    bool z[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int64_t k = k0 + (e < nk ? e : 0);
        c[e] = perm ? (int64_t)perm[k] : k;
        z[e] = dead && dead[c[e]];
    }
    const bool vec = (cols & 3) == 0;
    const int64_t r0 = (int64_t)blockIdx.y * IW_ROWS;
#pragma unroll
    for (int u = 0; u < IW_ROWS; ++u) {
        const int64_t r = r0 + u;
        if (r >= rows) break;
        const float* src = W + r * cols;
        float v[4];
        bool bad = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[e] = z[e] ? 0.0f : src[c[e]];
            bad |= !isfinite(v[e]);
        }
        if (bad) set_status(status, GPTQ_ERR_NONFINITE);
        float* dst = Wk + r * cols + k0;
        if (vec) {
            *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            for (int e = 0; e < nk; ++e) dst[e] = v[e];
        }
    }
}

// One warp per row: grid of Wk[r][c0:c1] -> cur_s/cur_z and the (scales, zeros) outputs.
__global__ void row_params_kernel(const float* __restrict__ Wk, int64_t rows, int64_t cols, int64_t c0, int64_t c1,
                                  int bits, int sym, int zr, float* __restrict__ cur_s, float* __restrict__ cur_z,
                                  float* __restrict__ scales, uint8_t* __restrict__ zeros, int64_t G, int64_t gi) {
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float* row = Wk + r * cols;
    float mx = -INFINITY, mn = INFINITY, am = 0.0f;
    for (int64_t c = c0 + lane; c < c1; c += 32) {
        const float v = row[c];
        mx = fmaxf(mx, v);
        mn = fminf(mn, v);
        am = fmaxf(am, fabsf(v));
    }
    Grid g;
    if (sym) {
        am = warp_max(am);
        g = sym_grid(am, (1 << (bits - 1)) - 1);
    } else {
        mx = warp_max(mx);
        mn = warp_min(mn);
        g = asym_grid(mn, mx, (1 << bits) - 1, zr != 0);
    }
    if (lane == 0) {
        cur_s[r] = g.s;
        cur_z[r] = g.z;
        scales[r * G + gi] = g.s;
        zeros[r * G + gi] = sym ? (uint8_t)(1 << (bits - 1)) : (uint8_t)g.z;
    }
}

struct BlockArgs {
    const float* Wk;
    int64_t rows, cols, j0;
    int bw;
    const float* U;
    int bits, sym, group;  // group in (0, 128] dividing 128: in-block params; else cur_s/cur_z
    int zr;                // asymmetric grid over a range widened to contain 0
    const float* cur_s;
    const float* cur_z;
    float* Err;
    float* ehi;  // optional TF32 split of Err (rows x QB, row stride eld)
    float* elo;
    int64_t eld;
    int8_t* codes;
    float* Wq;
    const int32_t* perm;
    float* scales;
    uint8_t* zeros;
    int64_t G;
    float* loss;
    int* status;
    int prune_k;        // pruning: weights pruned per row in this block
    uint8_t* mask;      // pruning: optional rows x cols mask output (original column order)
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// One 128-column block of the loop. TPR threads share a row; thread `sub` owns the
// 4-column chunks sub, sub+TPR, sub+2*TPR, ... of the block (CPT columns in registers),
// so the TPR lanes of a row read one contiguous 16*TPR-byte span of U's row per step.
// Besides its own chunks every lane keeps copies of the chunk being quantised (`cur`)
// and of the next one (`nxt`), updated with the same operations as the owner's, so the
// column-to-column dependency never goes through a shuffle: the next chunk is fetched
// from its owner one chunk ahead.
//
// PRUNE: the same loop with pruning in place of rounding (the GPTQ guide page's "Going
// further": SparseGPT reuses this update). At the block start each row ranks its block's
// saliencies (w_j / U[j][j])^2 of the updated weights (stable: ties by column) and prunes
// the a.prune_k smallest; then for every column q = 0 where pruned and q = w_j elsewhere
// (err = 0 there, so kept weights are left to the compensation of later columns).
template <int TPR, bool SMALL_GROUPS, bool PRUNE = false>
__global__ void __launch_bounds__(128) gptq_block_kernel(const BlockArgs a) {
    constexpr int CPT = QB / TPR;   // columns per thread
    constexpr int NCH = CPT / 4;    // 4-column chunks per thread
    constexpr int RPC = 128 / TPR;  // rows per CTA
    extern __shared__ __align__(16) float us[];  // QB x QB block of U, zeros below the diagonal
    __shared__ float invd[QB];

    // prologue (U is not written by any kernel of this call): U[blk, blk], upper part only
    const int bw = a.bw;
    const bool full = (bw == QB) && ((a.cols & 3) == 0);
    if (full) {
        const float* src = a.U + a.j0 * a.cols + a.j0;
#pragma unroll 8
        for (int v = threadIdx.x; v < QB * QB / 4; v += 128) {
            const int i = v >> 5, c4 = (v & 31) << 2;
            float* dst = us + i * QB + c4;
            if (c4 + 3 < i)
                *reinterpret_cast<float4*>(dst) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            else
                cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(dst)), src + i * a.cols + c4);
        }
        cp_async_wait_all();
        __syncthreads();
        // the chunk that straddles the diagonal: zero its part left of it
        for (int i = threadIdx.x; i < QB; i += 128)
            for (int c = i & ~3; c < i; ++c) us[i * QB + c] = 0.0f;
    } else {
#pragma unroll 4
        for (int idx = threadIdx.x; idx < QB * QB; idx += blockDim.x) {
            const int i = idx / QB, c = idx % QB;
            us[idx] = (i < bw && c < bw && c >= i) ? a.U[(a.j0 + i) * a.cols + a.j0 + c] : 0.0f;
        }
    }
    __syncthreads();
    bool u_bad = false;   // a diagonal entry of U that is not finite (reported after the wait)
    if (threadIdx.x < bw) {
        const float ujj = us[threadIdx.x * QB + threadIdx.x];
        u_bad = !isfinite(ujj);
        invd[threadIdx.x] = 1.0f / ujj;
    } else {
        invd[threadIdx.x] = 0.0f;
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    if (u_bad && blockIdx.x == 0) set_status(a.status, GPTQ_ERR_NONFINITE);

    const int sub = threadIdx.x % TPR;
    const int64_t row = (int64_t)blockIdx.x * RPC + threadIdx.x / TPR;
    const bool active = row < a.rows;
    const bool sym = a.sym != 0;
    const int qmax = sym ? (1 << (a.bits - 1)) - 1 : (1 << a.bits) - 1;
    const int lo = sym ? -qmax : 0, hi = qmax;
    const bool inblock_groups = a.group > 0 && a.group <= QB;

    // block column of this thread's element (m, e): chunk m*TPR + sub, element e
    auto col_of = [&](int m, int e) { return (m * TPR + sub) * 4 + e; };

    float w[CPT], er[CPT], qr[CPT];
    int8_t cr[CPT];
    const float* wrow = a.Wk + (active ? row : 0) * a.cols + a.j0;
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
        const int c0 = col_of(m, 0);
        if (full && active) {
            const float4 v = *reinterpret_cast<const float4*>(wrow + c0);
            w[4 * m] = v.x;
            w[4 * m + 1] = v.y;
            w[4 * m + 2] = v.z;
            w[4 * m + 3] = v.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) w[4 * m + e] = (active && c0 + e < bw) ? wrow[c0 + e] : 0.0f;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            er[4 * m + e] = 0.0f;
            qr[4 * m + e] = 0.0f;
            cr[4 * m + e] = 0;
        }
    }
    // grid of the group starting at block column jj (ending before gend), from the updated
    // weights: a TPR-lane reduction of max|w| (symmetric) or min/max (asymmetric)
    auto group_grid = [&](int jj, int gend) {
        float am = 0.0f, mx = -INFINITY, mn = INFINITY;
#pragma unroll
        for (int mm = 0; mm < NCH; ++mm)
#pragma unroll
            for (int ee = 0; ee < 4; ++ee) {
                const int c = col_of(mm, ee);
                if (c >= jj && c < gend) {
                    const float v = w[4 * mm + ee];
                    am = fmaxf(am, fabsf(v));
                    mx = fmaxf(mx, v);
                    mn = fminf(mn, v);
                }
            }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) {
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off, TPR));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off, TPR));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off, TPR));
        }
        const Grid gg = sym ? sym_grid(am, qmax) : asym_grid(mn, mx, qmax, a.zr != 0);
        if (active && sub == 0) {
            const int64_t gi = (a.j0 + jj) / a.group;
            a.scales[row * a.G + gi] = gg.s;
            a.zeros[row * a.G + gi] = sym ? (uint8_t)(1 << (a.bits - 1)) : (uint8_t)gg.z;
        }
        return gg;
    };

    // pruning: the row's mask over the block's 128 columns (bit c % 32 of word c / 32), the
    // same in every lane of the row
    uint32_t pm0 = 0u, pm1 = 0u, pm2 = 0u, pm3 = 0u;
    if constexpr (PRUNE) {
        float sal[CPT];
        int rank[CPT];
#pragma unroll
        for (int m = 0; m < NCH; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = col_of(m, e);
                const float t = w[4 * m + e] * (c < bw ? invd[c] : 0.0f);
                sal[4 * m + e] = c < bw ? t * t : INFINITY;
                rank[4 * m + e] = 0;
            }
        // rank of each own weight: how many of the block's weights come before it in the
        // stable ascending order of saliency (smaller, or equal at a lower column)
#pragma unroll
        for (int m = 0; m < NCH; ++m) {
#pragma unroll 1
            for (int o = 0; o < TPR; ++o) {
                if (4 * (m * TPR + o) >= bw) break;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 4 * (m * TPR + o) + e;
                    const float v = __shfl_sync(0xffffffffu, sal[4 * m + e], o, TPR);
                    if (c >= bw) continue;
#pragma unroll
                    for (int mm = 0; mm < NCH; ++mm)
#pragma unroll
                        for (int ee = 0; ee < 4; ++ee) {
                            const float sv = sal[4 * mm + ee];
                            rank[4 * mm + ee] += (v < sv || (v == sv && c < col_of(mm, ee))) ? 1 : 0;
                        }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < NCH; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = col_of(m, e);
                if (c < bw && rank[4 * m + e] < a.prune_k) {
                    const uint32_t bit = 1u << (c & 31);
                    const int wd = c >> 5;
                    pm0 |= wd == 0 ? bit : 0u;
                    pm1 |= wd == 1 ? bit : 0u;
                    pm2 |= wd == 2 ? bit : 0u;
                    pm3 |= wd == 3 ? bit : 0u;
                }
            }
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) {
            pm0 |= __shfl_xor_sync(0xffffffffu, pm0, off, TPR);
            pm1 |= __shfl_xor_sync(0xffffffffu, pm1, off, TPR);
            pm2 |= __shfl_xor_sync(0xffffffffu, pm2, off, TPR);
            pm3 |= __shfl_xor_sync(0xffffffffu, pm3, off, TPR);
        }
    }
    auto pruned = [&](int jj) -> bool {
        const int wd = jj >> 5;
        const uint32_t word = wd == 0 ? pm0 : wd == 1 ? pm1 : wd == 2 ? pm2 : pm3;
        return (word >> (jj & 31)) & 1u;
    };

    Grid g{1.0f, 1.0f, 0.0f};
    if (PRUNE) {
        // no grid
    } else if (!inblock_groups) {
        if (active) {
            g.s = a.cur_s[row];
            g.inv_s = 1.0f / g.s;
            g.z = a.cur_z[row];
        }
    } else if (!SMALL_GROUPS) {
        g = group_grid(0, bw);   // one group per block (group == 128)
    }
    float loss = 0.0f;
    int next_gs = 0;  // next in-block group start (groups smaller than the block)
    const float flo = (float)lo, fhi = (float)hi;

    // copies of chunk 0 (owner: lane 0, registers 0..3)
    float cur[4], nxt[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        cur[e] = __shfl_sync(0xffffffffu, w[e], 0, TPR);
        nxt[e] = 0.0f;
    }

    // one column step (chunk cc = m*TPR + o, element e): quantise cur[e], error, update
    // this thread's columns and both copies
    auto step = [&](int m, int o, int e, int jj) {
        const int cc = m * TPR + o;
        // shared-memory operands first, off the dependency chain
        const float* ur = us + jj * QB;
        const float id = invd[jj];
        const float4 uc = *reinterpret_cast<const float4*>(ur + 4 * cc);
        const float4 un = *reinterpret_cast<const float4*>(ur + min(4 * cc + 4, QB - 4));
        // this thread's chunks mm < m lie left of the current chunk for every lane (U is zero
        // there): neither loaded nor updated (m is a compile-time constant at each call)
        float4 uo[NCH];
#pragma unroll
        for (int mm = 0; mm < NCH; ++mm)
            if (mm >= m) uo[mm] = *reinterpret_cast<const float4*>(ur + col_of(mm, 0));
        const float wj = cur[e];
        float cf = 0.0f, q;
        if constexpr (PRUNE) {
            q = pruned(jj) ? 0.0f : wj;
        } else {
            cf = grid_code_f(wj, g, sym, flo, fhi);
            q = grid_dequant_f(cf, g, sym);
        }
        const float err = (wj - q) * id;
        if (sub == o) {
            cr[4 * m + e] = (int8_t)(int)cf;
            qr[4 * m + e] = q;
            er[4 * m + e] = err;
        }
        loss = fmaf(err, err, loss);
        if (e < 1) cur[1] = fmaf(-err, uc.y, cur[1]);
        if (e < 2) cur[2] = fmaf(-err, uc.z, cur[2]);
        if (e < 3) cur[3] = fmaf(-err, uc.w, cur[3]);
        nxt[0] = fmaf(-err, un.x, nxt[0]);
        nxt[1] = fmaf(-err, un.y, nxt[1]);
        nxt[2] = fmaf(-err, un.z, nxt[2]);
        nxt[3] = fmaf(-err, un.w, nxt[3]);
#pragma unroll
        for (int mm = 0; mm < NCH; ++mm) {
            if (mm < m) continue;
            const float4 u4 = uo[mm];
            w[4 * mm] = fmaf(-err, u4.x, w[4 * mm]);
            w[4 * mm + 1] = fmaf(-err, u4.y, w[4 * mm + 1]);
            w[4 * mm + 2] = fmaf(-err, u4.z, w[4 * mm + 2]);
            w[4 * mm + 3] = fmaf(-err, u4.w, w[4 * mm + 3]);
        }
    };

    // the owner lane o stays a runtime loop: a fully unrolled block (128 steps) overflows
    // the instruction cache
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
#pragma unroll 1
        for (int o = 0; o < TPR; ++o) {
            const int cc = m * TPR + o;
            if (4 * cc >= bw) break;
            // fetch the next chunk (m, o+1) or (m+1, 0) from its owner, current as of now
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = (o + 1 < TPR || m + 1 >= NCH) ? w[4 * m + e] : w[4 * (m + 1 < NCH ? m + 1 : m) + e];
                nxt[e] = __shfl_sync(0xffffffffu, v, (o + 1) % TPR, TPR);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int jj = 4 * cc + e;
                if (jj >= bw) break;
                if (!PRUNE && SMALL_GROUPS && jj == next_gs) {
                    next_gs += a.group;
                    g = group_grid(jj, min(jj + a.group, bw));
                }
                step(m, o, e, jj);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) cur[e] = nxt[e];
        }
    }
    (void)next_gs;

    if (!active) return;
    float* erow = a.Err + row * QB;
#pragma unroll
    for (int m = 0; m < NCH; ++m) {
        const int c0 = col_of(m, 0);
        *reinterpret_cast<float4*>(erow + c0) = make_float4(er[4 * m], er[4 * m + 1], er[4 * m + 2], er[4 * m + 3]);
        if (a.ehi) {
            float4 h, l;
            h.x = __uint_as_float(__float_as_uint(er[4 * m]) & 0xFFFFE000u);
            h.y = __uint_as_float(__float_as_uint(er[4 * m + 1]) & 0xFFFFE000u);
            h.z = __uint_as_float(__float_as_uint(er[4 * m + 2]) & 0xFFFFE000u);
            h.w = __uint_as_float(__float_as_uint(er[4 * m + 3]) & 0xFFFFE000u);
            l.x = er[4 * m] - h.x;
            l.y = er[4 * m + 1] - h.y;
            l.z = er[4 * m + 2] - h.z;
            l.w = er[4 * m + 3] - h.w;
            *reinterpret_cast<float4*>(a.ehi + row * a.eld + c0) = h;
            *reinterpret_cast<float4*>(a.elo + row * a.eld + c0) = l;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int lc = c0 + e;
            if (lc < bw) {
                const int64_t oc = a.perm ? (int64_t)a.perm[a.j0 + lc] : a.j0 + lc;
                if constexpr (PRUNE) {
                    if (a.mask) a.mask[row * a.cols + oc] = pruned(lc) ? 1 : 0;
                } else {
                    a.codes[row * a.cols + oc] = cr[4 * m + e];
                }
                if (a.Wq) a.Wq[row * a.cols + oc] = qr[4 * m + e];
            }
        }
    }
    if (sub == 0) a.loss[row] += loss;
}

__global__ void g_idx_kernel(const int32_t* __restrict__ perm, int64_t cols, int group, int32_t* __restrict__ g_idx) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= cols) return;
    const int64_t c = perm ? perm[k] : k;
    g_idx[c] = group ? (int32_t)(k / group) : 0;
}


// Rows whose length is a multiple of 32 codes: 32 codes fill exactly BITS words, so chunk c
// of the flat code array (codes 32c .. 32c+31, two 16-byte loads) becomes words
// BITS*c .. BITS*c+BITS-1 of the flat packed array (one 16- or 8-byte store for 4 and 2
// bits, three 4-byte stores for 3). Grid-stride over the chunks; each byte is read once and
// each word written once, with streaming cache hints.
template <int BITS>
__global__ void __launch_bounds__(256) pack32_kernel(const int8_t* __restrict__ codes, int64_t chunks, int offset,
                                                     uint32_t* __restrict__ packed) {
    constexpr uint32_t mask = (1u << BITS) - 1u;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks;
         c += (int64_t)gridDim.x * blockDim.x) {
        const int4* src = reinterpret_cast<const int4*>(codes) + 2 * c;
        const int4 v0 = __ldcs(src), v1 = __ldcs(src + 1);
        const uint32_t b[8] = {(uint32_t)v0.x, (uint32_t)v0.y, (uint32_t)v0.z, (uint32_t)v0.w,
                               (uint32_t)v1.x, (uint32_t)v1.y, (uint32_t)v1.z, (uint32_t)v1.w};
        uint32_t w[BITS];
#pragma unroll
        for (int k = 0; k < BITS; ++k) w[k] = 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            // the low BITS bits of (code byte + offset): carries out of the byte are masked off
            const uint32_t u = ((b[i >> 2] >> (8 * (i & 3))) + (uint32_t)offset) & mask;
            const int pos = i * BITS;
            w[pos >> 5] |= u << (pos & 31);
            if ((pos & 31) + BITS > 32) w[(pos >> 5) + 1] |= u >> (32 - (pos & 31));
        }
        uint32_t* dst = packed + (int64_t)BITS * c;
        if constexpr (BITS == 4) {
            __stcs(reinterpret_cast<uint4*>(dst), make_uint4(w[0], w[1], w[2], w[3]));
        } else if constexpr (BITS == 2) {
            __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w[0], w[1]));
        } else {
#pragma unroll
            for (int k = 0; k < BITS; ++k) __stcs(dst + k, w[k]);
        }
    }
}

// One thread per output word: bits [32w, 32w+32) of the row's LSB-first b-bit stream (any
// row length and alignment).
__global__ void pack_kernel(const int8_t* __restrict__ codes, int64_t rows, int64_t cols, int bits, int offset,
                            int64_t words, uint32_t* __restrict__ packed) {
    const int64_t r = blockIdx.y;
    const uint32_t mask = (1u << bits) - 1u;
    for (int64_t wd = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; wd < words; wd += (int64_t)gridDim.x * blockDim.x) {
        const int64_t bit0 = wd * 32;
        const int64_t c0 = bit0 / bits;
        const int64_t c1 = std::min<int64_t>(cols - 1, (bit0 + 31) / bits);
        uint64_t acc = 0;
        for (int64_t c = c0; c <= c1; ++c) {
            const uint32_t u = (uint32_t)((int)codes[r * cols + c] + offset) & mask;
            const int64_t pos = c * bits - bit0;
            acc |= pos >= 0 ? ((uint64_t)u << pos) : ((uint64_t)u >> (-pos));
        }
        packed[r * words + wd] = (uint32_t)acc;
    }
}

// Round-to-nearest: one warp per (row, group) (group > 0) or one CTA per row (group == 0).
// A weight that is not finite (outside a dead column) records GPTQ_ERR_NONFINITE.
__global__ void rtn_group_kernel(const float* __restrict__ W, int64_t rows, int64_t cols, const uint8_t* __restrict__ dead,
                                 int bits, int sym, int zr, int group, int64_t G, int8_t* __restrict__ codes,
                                 float* __restrict__ scales, uint8_t* __restrict__ zeros, float* __restrict__ Wq,
                                 int* __restrict__ status) {
    const int64_t task = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (task >= rows * G) return;
    const int64_t r = task / G, gi = task % G;
    const int64_t c0 = gi * group, c1 = std::min<int64_t>(cols, c0 + group);
    const float* row = W + r * cols;
    float mx = -INFINITY, mn = INFINITY, am = 0.0f;
    bool bad = false;
    for (int64_t c = c0 + lane; c < c1; c += 32) {
        const float v = (dead && dead[c]) ? 0.0f : row[c];
        bad |= !isfinite(v);
        mx = fmaxf(mx, v);
        mn = fminf(mn, v);
        am = fmaxf(am, fabsf(v));
    }
    if (bad) set_status(status, GPTQ_ERR_NONFINITE);
    const int qmax = sym ? (1 << (bits - 1)) - 1 : (1 << bits) - 1;
    const Grid g = sym ? sym_grid(warp_max(am), qmax) : asym_grid(warp_min(mn), warp_max(mx), qmax, zr != 0);
    if (lane == 0) {
        scales[r * G + gi] = g.s;
        zeros[r * G + gi] = sym ? (uint8_t)(1 << (bits - 1)) : (uint8_t)g.z;
    }
    const int lo = sym ? -qmax : 0;
    for (int64_t c = c0 + lane; c < c1; c += 32) {
        const float v = (dead && dead[c]) ? 0.0f : row[c];
        const int code = grid_code(v, g, sym != 0, lo, qmax);
        codes[r * cols + c] = (int8_t)code;
        if (Wq) Wq[r * cols + c] = grid_dequant(code, g, sym != 0);
    }
}

__global__ void __launch_bounds__(256) rtn_row_kernel(const float* __restrict__ W, int64_t rows, int64_t cols,
                                                     const uint8_t* __restrict__ dead, int bits, int sym, int zr,
                                                     int8_t* __restrict__ codes, float* __restrict__ scales,
                                                     uint8_t* __restrict__ zeros, float* __restrict__ Wq,
                                                     int* __restrict__ status) {
    const int64_t r = blockIdx.x;
    const float* row = W + r * cols;
    __shared__ float red[3][8];
    float mx = -INFINITY, mn = INFINITY, am = 0.0f;
    bool bad = false;
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) {
        const float v = (dead && dead[c]) ? 0.0f : row[c];
        bad |= !isfinite(v);
        mx = fmaxf(mx, v);
        mn = fminf(mn, v);
        am = fmaxf(am, fabsf(v));
    }
    if (bad) set_status(status, GPTQ_ERR_NONFINITE);
    mx = warp_max(mx);
    mn = warp_min(mn);
    am = warp_max(am);
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[0][wid] = mx;
        red[1][wid] = mn;
        red[2][wid] = am;
    }
    __syncthreads();
    mx = -INFINITY;
    mn = INFINITY;
    am = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
        mx = fmaxf(mx, red[0][i]);
        mn = fminf(mn, red[1][i]);
        am = fmaxf(am, red[2][i]);
    }
    const int qmax = sym ? (1 << (bits - 1)) - 1 : (1 << bits) - 1;
    const Grid g = sym ? sym_grid(am, qmax) : asym_grid(mn, mx, qmax, zr != 0);
    if (threadIdx.x == 0) {
        scales[r] = g.s;
        zeros[r] = sym ? (uint8_t)(1 << (bits - 1)) : (uint8_t)g.z;
    }
    const int lo = sym ? -qmax : 0;
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) {
        const float v = (dead && dead[c]) ? 0.0f : row[c];
        const int code = grid_code(v, g, sym != 0, lo, qmax);
        codes[r * cols + c] = (int8_t)code;
        if (Wq) Wq[r * cols + c] = grid_dequant(code, g, sym != 0);
    }
}

int launch_pack(const int8_t* codes, int64_t rows, int64_t cols, int bits, int sym, uint32_t* packed, cudaStream_t s) {
    const int offset = sym ? (1 << (bits - 1)) : 0;
    if (cols % 32 == 0 && (reinterpret_cast<uintptr_t>(codes) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(packed) & 15) == 0) {
        const int64_t chunks = rows * (cols / 32);
        const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(chunks, 256), (int64_t)device_sm_count() * 8);
        switch (bits) {
            case 2: GPTQ_LAUNCH(K_PACK, s, pack32_kernel<2><<<grid, 256, 0, s>>>(codes, chunks, offset, packed)); break;
            case 3: GPTQ_LAUNCH(K_PACK, s, pack32_kernel<3><<<grid, 256, 0, s>>>(codes, chunks, offset, packed)); break;
            default: GPTQ_LAUNCH(K_PACK, s, pack32_kernel<4><<<grid, 256, 0, s>>>(codes, chunks, offset, packed)); break;
        }
        GPTQ_LAUNCH_CHECK();
        return GPTQ_OK;
    }
    const int64_t words = gptq_packed_words_per_row(cols, bits);
    const unsigned gx = (unsigned)std::min<int64_t>(ceil_div(words, 256), 1024);
    dim3 grid(gx, (unsigned)rows);
    GPTQ_LAUNCH(K_PACK, s, pack_kernel<<<grid, 256, 0, s>>>(codes, rows, cols, bits, sym ? (1 << (bits - 1)) : 0, words, packed));
    GPTQ_LAUNCH_CHECK();
    return GPTQ_OK;
}

}  // namespace
}  // namespace gptq

using namespace gptq;

extern "C" int64_t gptq_packed_words_per_row(int64_t cols, int bits) {
    if (cols < 0 || bits < 1 || bits > 8) return 0;
    return (cols * bits + 31) / 32;
}

extern "C" size_t gptq_quantize_workspace_bytes(int64_t rows, int64_t cols, gptq_qconfig q) {
    (void)q;
    if (rows <= 0 || cols <= 0) return 0;
    return carve(nullptr, rows, cols).bytes;
}

extern "C" int gptq_pack(const int8_t* codes, int64_t rows, int64_t cols, int bits, int sym, uint32_t* packed,
                         void* stream) {
    if (rows < 0 || cols < 0) return GPTQ_ERR_INVALID_ARG;
    if (bits < 2 || bits > 4) return GPTQ_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return GPTQ_OK;
    if (!codes || !packed || rows > 65535) return GPTQ_ERR_INVALID_ARG;
    return launch_pack(codes, rows, cols, bits, sym, packed, static_cast<cudaStream_t>(stream));
}

namespace gptq {
namespace {

// The column loop shared by gptq_quantize and gptq_prune (prune_sparsity < 0: quantize).
int column_loop(const float* W, int64_t rows, int64_t cols, const float* U, const int32_t* perm,
                const uint8_t* dead, gptq_qconfig q, int8_t* codes, float* scales, uint8_t* zeros, int32_t* g_idx,
                float* Wq, uint32_t* packed, float* row_loss, void* ws, size_t ws_bytes, void* stream,
                double prune_sparsity, uint8_t* mask) {
    const bool prune = prune_sparsity >= 0.0;
    QuantWs w = carve(ws, rows, cols);
    if (ws_bytes < w.bytes) return GPTQ_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t G = (!prune && q.group) ? ceil_div(cols, q.group) : 1;

    // (the memsets first: every later item in the stream is one of this call's kernels, so
    // the block and trailing kernels may be launched as programmatic dependents)
    // the per-row loss accumulates straight into the caller's row_loss when given
    float* loss = row_loss ? row_loss : w.loss;
    GPTQ_CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(float) * rows, s));
    GPTQ_CUDA_TRY(cudaMemsetAsync(w.status, 0, sizeof(int), s));
    {
        dim3 grid((unsigned)ceil_div(cols, 4 * 256), (unsigned)ceil_div(rows, IW_ROWS));
        GPTQ_LAUNCH(K_INIT_WORK, s, init_work_kernel<<<grid, 256, 0, s>>>(W, rows, cols, perm, dead, w.W, w.status));
        GPTQ_LAUNCH_CHECK();
    }
    // tensor-core trailing update when every row of W and U is 16-byte aligned
    const bool tc = (cols % 4 == 0) && tc_gemm_nt_ok(w.W, cols);
    // U^T's split: the trailing updates read it strictly below the diagonal only (rows past
    // the block, the block's columns), so the tiles with nothing there are skipped
    if (tc) GPTQ_CUDA_TRY(split_cols(K_SPLIT, U, cols, (int)cols, (int)cols, w.uhi, w.ulo, (int)cols, s, false, true));
    const unsigned pgrid = (unsigned)ceil_div(rows, 8);
    if (!prune && q.group == 0) {
        GPTQ_LAUNCH(K_ROW_PARAMS, s, row_params_kernel<<<pgrid, 256, 0, s>>>(w.W, rows, cols, 0, cols, q.bits, q.sym, q.zero_in_range,
                                                                             w.cur_s, w.cur_z, scales, zeros, G, 0));
        GPTQ_LAUNCH_CHECK();
    }

    // threads per row: as many as keep every CTA resident at once (3 per SM: 64.5 KB of
    // shared memory and at most 128 threads x 167 registers each)
    const int sms = device_sm_count();
    int tpr = 4;
    for (int t : {32, 16, 8}) {
        if (ceil_div(rows * t, 128) <= 3 * sms) {
            tpr = t;
            break;
        }
    }
    const size_t smem = sizeof(float) * QB * QB;
    const bool small_groups = !prune && q.group > 0 && q.group < QB;
    auto block_fn = [&](int t) -> void (*)(BlockArgs) {
        if (prune) {
            switch (t) {
                case 32: return gptq_block_kernel<32, false, true>;
                case 16: return gptq_block_kernel<16, false, true>;
                case 8: return gptq_block_kernel<8, false, true>;
                default: return gptq_block_kernel<4, false, true>;
            }
        }
        switch (t) {
            case 32: return small_groups ? gptq_block_kernel<32, true> : gptq_block_kernel<32, false>;
            case 16: return small_groups ? gptq_block_kernel<16, true> : gptq_block_kernel<16, false>;
            case 8: return small_groups ? gptq_block_kernel<8, true> : gptq_block_kernel<8, false>;
            default: return small_groups ? gptq_block_kernel<4, true> : gptq_block_kernel<4, false>;
        }
    };
    void (*kblock)(BlockArgs) = block_fn(tpr);
    GPTQ_CUDA_TRY(cudaFuncSetAttribute(kblock, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    BlockArgs a{};
    a.Wk = w.W;
    a.rows = rows;
    a.cols = cols;
    a.U = U;
    a.bits = q.bits;
    a.sym = q.sym;
    a.zr = q.zero_in_range;
    a.group = prune ? 0 : q.group;
    a.cur_s = w.cur_s;
    a.cur_z = w.cur_z;
    a.Err = w.Err;
    const int SB = super_blocks(cols);
    a.eld = SB * QB;
    a.codes = codes;
    a.Wq = Wq;
    a.perm = perm;
    a.scales = scales;
    a.zeros = zeros;
    a.G = G;
    a.loss = loss;
    a.status = w.status;
    a.mask = mask;
    const unsigned bgrid = (unsigned)ceil_div(rows, 128 / tpr);
    for (int64_t j0 = 0; j0 < cols; j0 += QB) {
        const int bw = (int)std::min<int64_t>(QB, cols - j0);
        if (!prune && q.group > QB && j0 % q.group == 0) {
            GPTQ_LAUNCH(K_ROW_PARAMS, s,
                        row_params_kernel<<<pgrid, 256, 0, s>>>(w.W, rows, cols, j0,
                                                                std::min<int64_t>(cols, j0 + q.group), q.bits, q.sym,
                                                                q.zero_in_range,
                                                                w.cur_s, w.cur_z, scales, zeros, G, j0 / q.group));
            GPTQ_LAUNCH_CHECK();
        }
        a.j0 = j0;
        a.bw = bw;
        // pruning: round(sparsity * width), ties to even, in double
        a.prune_k = prune ? (int)std::nearbyint(prune_sparsity * (double)bw) : 0;
        // this block's errors go to its slot of the super-block's split
        const int64_t sb0 = j0 / (SB * QB) * (SB * QB), sb_end = std::min<int64_t>(cols, sb0 + SB * QB);
        a.ehi = tc ? w.ehi + (j0 - sb0) : nullptr;
        a.elo = tc ? w.elo + (j0 - sb0) : nullptr;
        cudaError_t le = cudaSuccess;
        GPTQ_LAUNCH(K_BLOCK, s, le = launch_pdl(kblock, dim3(bgrid), dim3(128), smem, s, a));
        GPTQ_CUDA_TRY(le);
        GPTQ_LAUNCH_CHECK();
        const int64_t e = j0 + bw;
        if (e < cols) {
            if (tc) {
                // W[:, e:] -= Err * U[blk, e:] = Err * (U^T[e:, blk])^T on the tensor cores,
                // deferred for the columns past the super-block: inside it only the block's
                // own super-block columns are updated (K = 128); at its end the columns past
                // it take the errors of all its blocks at once (K = SB * 128), so the large
                // trailing matrix is read and written once per SB blocks.
                GemmOpts o;
                o.ldb = cols;
                o.pdl = true;
                o.narrow_ok = true;   // on the loop's critical path: 128x64 tiles when they fit one wave
                if (e < sb_end) {
                    GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_TRAIL, (int)rows, (int)(sb_end - e), bw, -1.0f, w.ehi + (j0 - sb0),
                                             w.elo + (j0 - sb0), w.uhi + e * cols + j0, w.ulo + e * cols + j0, SB * QB,
                                             1.0f, w.W + e, cols, false, w.status, s, o));
                } else {
                    GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_TRAIL, (int)rows, (int)(cols - e), (int)(e - sb0), -1.0f, w.ehi,
                                             w.elo, w.uhi + e * cols + sb0, w.ulo + e * cols + sb0, SB * QB, 1.0f,
                                             w.W + e, cols, false, w.status, s, o));
                }
            } else {
                GPTQ_CUDA_TRY(sgemm(K_SGEMM_TRAIL, false, (int)rows, (int)(cols - e), bw, -1.0f, w.Err, QB,
                                    U + j0 * cols + e, cols, 1.0f, w.W + e, cols, false, s));
            }
        }
    }

    if (g_idx) {
        GPTQ_LAUNCH(K_G_IDX, s, g_idx_kernel<<<(unsigned)ceil_div(cols, 256), 256, 0, s>>>(perm, cols, q.group, g_idx));
        GPTQ_LAUNCH_CHECK();
    }
    if (packed) {
        const int rc = launch_pack(codes, rows, cols, q.bits, q.sym, packed, s);
        if (rc != GPTQ_OK) return rc;
    }
    return finish_call(w.status, s);
}

}  // namespace
}  // namespace gptq

extern "C" int gptq_quantize(const float* W, int64_t rows, int64_t cols, const float* U, const int32_t* perm,
                             const uint8_t* dead, gptq_qconfig q, int8_t* codes, float* scales, uint8_t* zeros,
                             int32_t* g_idx, float* Wq, uint32_t* packed, float* row_loss, void* ws, size_t ws_bytes,
                             void* stream) {
    if (rows < 0 || cols < 0) return GPTQ_ERR_INVALID_ARG;
    if (q.bits < 2 || q.bits > 4 || !group_ok(q.group)) return GPTQ_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return GPTQ_OK;
    if (!W || !U || !codes || !scales || !zeros || !ws || rows > 65535) return GPTQ_ERR_INVALID_ARG;
    return column_loop(W, rows, cols, U, perm, dead, q, codes, scales, zeros, g_idx, Wq, packed, row_loss, ws,
                       ws_bytes, stream, -1.0, nullptr);
}

extern "C" size_t gptq_prune_workspace_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return carve(nullptr, rows, cols).bytes;
}

extern "C" int gptq_prune(const float* W, int64_t rows, int64_t cols, const float* U, const int32_t* perm,
                          const uint8_t* dead, float sparsity, float* Wp, uint8_t* mask, float* row_loss, void* ws,
                          size_t ws_bytes, void* stream) {
    if (rows < 0 || cols < 0) return GPTQ_ERR_INVALID_ARG;
    if (!(sparsity >= 0.0f && sparsity <= 1.0f)) return GPTQ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return GPTQ_OK;
    if (!W || !U || !Wp || !ws || rows > 65535) return GPTQ_ERR_INVALID_ARG;
    gptq_qconfig q{4, 0, 1, 0};   // unused by the pruning loop
    return column_loop(W, rows, cols, U, perm, dead, q, nullptr, nullptr, nullptr, nullptr, Wp, nullptr, row_loss,
                       ws, ws_bytes, stream, (double)sparsity, mask);
}

extern "C" int rtn_quantize(const float* W, int64_t rows, int64_t cols, const uint8_t* dead, gptq_qconfig q,
                            int8_t* codes, float* scales, uint8_t* zeros, float* Wq, uint32_t* packed, void* stream) {
    if (rows < 0 || cols < 0) return GPTQ_ERR_INVALID_ARG;
    if (q.bits < 2 || q.bits > 4 || q.group < 0) return GPTQ_ERR_UNSUPPORTED;
    if (rows == 0 || cols == 0) return GPTQ_OK;
    if (!W || !codes || !scales || !zeros || rows > 65535) return GPTQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the call's status word (static device memory, cleared on the stream: no allocation)
    int* status = nullptr;
    GPTQ_CUDA_TRY(call_status_word(s, &status));
    if (q.group == 0) {
        GPTQ_LAUNCH(K_RTN, s, rtn_row_kernel<<<(unsigned)rows, 256, 0, s>>>(W, rows, cols, dead, q.bits, q.sym,
                                                                             q.zero_in_range, codes, scales, zeros,
                                                                             Wq, status));
    } else {
        const int64_t G = ceil_div(cols, q.group);
        const int64_t tasks = rows * G;
        GPTQ_LAUNCH(K_RTN, s,
                    rtn_group_kernel<<<(unsigned)ceil_div(tasks, 8), 256, 0, s>>>(W, rows, cols, dead, q.bits, q.sym,
                                                                                  q.zero_in_range, q.group, G, codes,
                                                                                  scales, zeros, Wq, status));
    }
    GPTQ_LAUNCH_CHECK();
    if (packed) {
        const int rc = launch_pack(codes, rows, cols, q.bits, q.sym, packed, s);
        if (rc != GPTQ_OK) return rc;
    }
    return finish_call(status, s);
}

extern "C" const char* gptq_status_string(int status) {
    switch (status) {
        case GPTQ_OK: return "ok";
        case GPTQ_ERR_INVALID_ARG: return "invalid argument";
        case GPTQ_ERR_UNSUPPORTED: return "unsupported configuration";
        case GPTQ_ERR_NOT_SPD: return "Hessian not positive definite (Cholesky pivot <= 0)";
        case GPTQ_ERR_CUDA: return "CUDA error";
        case GPTQ_ERR_TIMEOUT: return "on-device wait timed out";
        case GPTQ_ERR_WORKSPACE: return "workspace too small";
        case GPTQ_ERR_NONFINITE: return "input not finite (NaN or infinity)";
        default: return "unknown status";
    }
}
