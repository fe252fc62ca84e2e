// tcgen05 GEMM for the projections around the attention (sm_103a, bf16, fp32 accumulation).
//
//   absorb: q_cat[n, h, c] = sum_j W_UK[c, h*d_h + j] * q_nope[n, h, j]      (M = c, K = j)
//   out:    o[n, h*d_h + j] = sum_c W_UV[c, h*d_h + j] * o_lat[n, h, c]       (M = j, K = c)
//   append: row[n, c] = sum_k [W_DKV | W_KR][k, c] * x[n, k], stored to the paged pool with
//           RoPE(., pos[n]) on the last d_r columns                            (M = c, K = k)
//   oproj:  out[n, m] = sum_k W_O[k, m] * o[n, k], k over n_h*d_h               (M = m, K = k)
//   absorbc: q_cat[n, h, c] = sum_k W_UQK[k, h*d_c + c] * c_q[n, k], the absorbed query from the
//           compressed query latent with W_UQ folded into W_UK (RoPE half as in absorb) (M = c, K = k)
//
// All are computed "weights as M, tokens as N": D[m, n] = sum_k A[m, k] * B[n, k] with a
// 128-row weight tile as A (K-major for W_UK, MN-major for W_UV, W_DKV, W_KR and W_O, as the
// weights are stored) and up to 256 tokens as B (K-major).  Each CTA owns one m-tile of up to
// HPC heads for one n-tile: warp 0 streams 64-wide K chunks of A and B through a ring that
// fills shared memory, warp 1 issues the MMAs into one TMEM accumulator per head, warps 2-5
// drain D (one row per thread).  With few tokens (decode) a CTA's whole weight slice is in
// flight at once.  The kernel is launched as a programmatic dependent: the weights do not
// depend on the previous kernel, so their loads are issued before the grid-dependency wait and
// only the token operand after it.  In ABSORB mode the CTAs also write the RoPE half of q_cat
// (RoPE(q_rope[n, h], pos[n]) into columns [d_c, d_c + d_r)), spread over all CTAs of a token
// tile, with the epilogue warps, which are idle while the weights stream.  A deep K (APPEND's
// d_model, OPROJ's n_h*d_h) over too few output tiles is split over a cluster of CTAs that add
// their partial sums through distributed shared memory.  Each mode is its own instantiation.
#pragma once

#include <cudaTypedefs.h>

#include "mx_format.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tcg {

constexpr int BM = 128, BK = 64, MAX_N = 256, HPC = 4, MAX_STAGES = 16;
constexpr int MAX_KSPLIT = 8;                 // portable cluster size
constexpr int SPLIT_STAGES = 3;               // ring depth of split-K CTAs (several share an SM)
constexpr int SPLIT_BELOW_CTAS = 148;         // fewer output tiles than SMs: split K
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int NTHREADS = 192;
constexpr int SMEM_LIMIT = 232448;            // opt-in shared memory per CTA

// stage = A tile + B tile (n_pad rows of 128 B), rounded to the 1 KB swizzle atom
__host__ __device__ inline int stage_bytes(int n_pad) { return (A_BYTES + n_pad * BK * 2 + 1023) & ~1023; }
// ring, barriers, TMEM slot, then (APPEND) the pool row offset of each token of the tile
__host__ __device__ inline int smem_bytes(int n_pad, int stages) { return stages * stage_bytes(n_pad) + 16 * stages + 48 + 4 * MAX_N; }
__host__ __device__ inline uint32_t tmem_cols(int n_pad) {
    uint32_t c = 32;
    while ((int)c < n_pad) c <<= 1;
    return c;
}
// Ring depth.  Few tokens: at most three stages (and no more than the chunks a CTA streams), so
// that several CTAs share an SM (measured on B300: the weight streams gain from more resident
// CTAs, not from a deeper ring per CTA).  Many tokens: as deep as shared memory allows.
inline int max_stages(int n_pad) {
    int s = (SMEM_LIMIT - 48 - 4 * MAX_N) / (stage_bytes(n_pad) + 16);
    return s < MAX_STAGES ? s : MAX_STAGES;
}
inline int stages_for(int n_pad) {
    const int s = max_stages(n_pad);
    return n_pad <= 64 && s > 3 ? 3 : s;
}
// Heads per CTA (one TMEM accumulator of tmem_cols(n_pad) columns each, <= 512 columns in all).
// One by default: more CTAs stream the weights faster than fewer CTAs with more heads each.
inline int max_heads_per_cta(int n_pad) {
    int h = 512 / (int)tmem_cols(n_pad);
    return h < HPC ? h : HPC;
}

enum Mode { ABSORB = 0, OUT = 1, APPEND = 2, OPROJ = 3, ABSORBC = 4 };

struct GemmArgs {
    int mode;
    int n_tokens;       // valid tokens
    int n_pad;          // MMA N (multiple of 16, >= 16, <= 256)
    int k_chunks;       // K / 64
    int n_h, d_h, d_c, width;
    int stages;         // ring depth
    int hpc;            // heads per CTA
    void* out;          // q_cat (ABSORB) or o (OUT), bf16
    unsigned long long wait_ns;
    // ABSORB: the RoPE half (q_rope [n, n_h, d_r] bf16 unrotated, pos [n]); q_rope may be null
    const bf16* q_rope;
    const int* pos;
    int d_r;
    RopeFreq rf;
    int n_tile;         // tokens per CTA tile (the grid's z dimension walks them)
    int ksplit;         // K split over a cluster of this many CTAs (1: none; > 1 needs hpc 1)
    // APPEND: the paged pool and where each token goes (pos is the token's position)
    void* pool;
    const int* page_table;
    const int* seq_idx;
    int max_pages, batch, page_size;
    long long num_pages;
    int kv_format;      // APPEND: KV_PLAIN rows of bf16, or an MX cache (codes in pool)
    void* scales;       // APPEND, MX cache: [num_pages, P, W / 32] scale bytes
};

// APPEND into an MX cache: the warp's 32 lanes hold one token's values of the block of 32
// columns that starts at column cb (lane l: column cb + l) of cache row `ro` (ro < 0: a token
// that goes nowhere; the warp still takes part in the shuffles).
__device__ __forceinline__ void mx_append_block(const GemmArgs& g, int ro, int cb, float v, int lane) {
    const int r = ro < 0 ? 0 : ro;
    uint8_t* scale = reinterpret_cast<uint8_t*>(g.scales) + (size_t)r * (g.width / MX_BLOCK) + cb / MX_BLOCK;
    if (g.kv_format == KV_MXFP8)
        mx_store_block<KV_MXFP8>(reinterpret_cast<uint8_t*>(g.pool) + (size_t)r * g.width + cb, scale, v, lane, ro >= 0);
    else
        mx_store_block<KV_MXFP4>(reinterpret_cast<uint8_t*>(g.pool) + (size_t)r * (g.width / 2) + cb / 2, scale, v,
                                 lane, ro >= 0);
}

// launch choices (0 = automatic), from the library's tuning knobs
struct Tuning {
    unsigned long long wait_ns = 2000000000ull;
    int hpc = 0, stages = 0, ksplit = 0;
    bool pdl = true;
};

__device__ __forceinline__ bool gwait(uint32_t bar, uint32_t parity, unsigned long long limit) {
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (i & 1u) {  // every second failed poll (try_wait itself may suspend the thread)
            const unsigned long long t = globaltimer_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > limit) {
                set_device_error(MLA_ERR_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

// Chunk c of a CTA with nh heads and kper K chunks per head: head-major for ABSORB (a head's K
// chunks are adjacent columns of W_UK), K-major for OUT (the CTA's heads are adjacent column
// slabs of W_UV, so one 64-row block of all of them is requested together).  chunk_k is the
// index within the CTA's K range.
template <int MODE>
__device__ __forceinline__ int chunk_head(int c, int nh, int kper) {
    return (MODE == OUT || MODE == ABSORBC) ? c % nh : c / kper;
}
template <int MODE>
__device__ __forceinline__ int chunk_k(int c, int nh, int kper) {
    return (MODE == OUT || MODE == ABSORBC) ? c / nh : c % kper;
}

// Pool row (element offset) of appended token n, or -1 (and the bounds error) when its sequence,
// position or page is outside the cache.
__device__ __forceinline__ long long append_row(const GemmArgs& g, int n) {
    const int b = __ldg(g.seq_idx + n), p = __ldg(g.pos + n);
    if (b < 0 || b >= g.batch || p < 0 || p >= g.max_pages * g.page_size) {
        set_device_error(MLA_ERR_DEVICE_BOUNDS);
        return -1;
    }
    const int page = __ldg(g.page_table + (long long)b * g.max_pages + p / g.page_size);
    if (page < 0 || page >= g.num_pages) {
        set_device_error(MLA_ERR_DEVICE_BOUNDS);
        return -1;
    }
    return ((long long)page * g.page_size + p % g.page_size) * g.width;
}

// ABSORB: the RoPE half of q_cat for the tokens of this CTA's n-tile, shared among all the
// tile's CTAs.  The tile's (token, pair) items are cut into equal runs, one per CTA; a thread
// takes items of its CTA's run and rotates each for a strided subset of the heads, so that the
// cos and sin of an angle are computed once per CTA rather than once per head.  tid: 0..127.
__device__ __forceinline__ void absorb_rope(const GemmArgs& g, int n0, int tid) {
    const int half = g.d_r / 2;
    const int items = min(g.n_tile, g.n_tokens - n0) * half;
    const int ctas = (int)(gridDim.x * gridDim.y), cta = (int)(blockIdx.y * gridDim.x + blockIdx.x);
    const int per = (items + ctas - 1) / ctas;
    const int p0 = cta * per, np = min(per, items - p0);
    if (np <= 0) return;
    const int G = np < 128 ? np : 128;   // threads per head group
    const int HG = 128 / G, hg = tid / G;
    if (hg >= HG) return;
    bf16* qc = reinterpret_cast<bf16*>(g.out);
    constexpr int BATCH = 8;  // loads in flight per thread before the first store
    for (int q = p0 + tid % G; q < p0 + np; q += G) {
        const int n = n0 + q / half, i = q % half;
        float c, sn;
        rope_cos_sin(__ldg(g.pos + n), g.rf.theta[i], &c, &sn);
        const uint32_t* src = reinterpret_cast<const uint32_t*>(g.q_rope + (size_t)n * g.n_h * g.d_r + 2 * i);
        for (int h = hg; h < g.n_h; h += HG * BATCH) {
            uint32_t x[BATCH];
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                const int hh = h + j * HG;
                x[j] = hh < g.n_h ? __ldg(src + (size_t)hh * (g.d_r / 2)) : 0u;
            }
#pragma unroll
            for (int j = 0; j < BATCH; ++j) {
                const int hh = h + j * HG;
                if (hh >= g.n_h) break;
                const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&x[j]);
                const float x0 = __bfloat162float(v.x), x1 = __bfloat162float(v.y);
                *reinterpret_cast<__nv_bfloat162*>(qc + ((size_t)n * g.n_h + hh) * g.width + g.d_c + 2 * i) =
                    __floats2bfloat162_rn(x0 * c - x1 * sn, x0 * sn + x1 * c);
            }
        }
    }
}

// The 32 lanes of a warp hold one token's values of 32 consecutive latent columns (lane l:
// column c0 + l).  Each group of 8 lanes packs its values to bf16 (round to nearest even, as a
// single conversion would) and its first lane stores them as one 16-byte store at dst, its own
// column's address (8-column aligned).  All lanes take part in the shuffles; `store` gates the
// write (warp-uniform).
__device__ __forceinline__ void store_cols8(bf16* dst, float v, int lane, bool store) {
    const float nb = __shfl_down_sync(0xffffffffu, v, 1);
    const uint32_t pair = ptx::pack_bf16(v, nb);  // meaningful in even lanes
    const uint32_t p1 = __shfl_down_sync(0xffffffffu, pair, 2);
    const uint32_t p2 = __shfl_down_sync(0xffffffffu, pair, 4);
    const uint32_t p3 = __shfl_down_sync(0xffffffffu, pair, 6);
    if (store && (lane & 7) == 0) *reinterpret_cast<uint4*>(dst) = make_uint4(pair, p1, p2, p3);
}

// Split K: the CTA of cluster rank ks adds the partial sums of all ksplit CTAs (in rank order,
// so the result does not depend on timing) for its slice of the tile's tokens and stores them
// as the mode's epilogue would.  Partials sit at the start of each CTA's shared memory as
// [n_pad][128] fp32; tid (0..127) is the row m of the tile.
template <int MODE>
__device__ __forceinline__ void split_store(const GemmArgs& g, uint32_t base, const int* rowoff, int mt, int h0,
                                            int n0, int ks, bool rope_tile, int tid) {
    const int KS = g.ksplit;
    const int n_here = min(g.n_pad, g.n_tokens - n0);
    const int per = (n_here + KS - 1) / KS, t0 = ks * per, t1 = min(n_here, t0 + per);
    bf16* out = reinterpret_cast<bf16*>(MODE == APPEND ? g.pool : g.out);
    for (int nl = t0; nl < t1; ++nl) {
        const uint32_t a = base + (uint32_t)(nl * BM + tid) * 4u;
        // four ranks' loads in flight per add round; the sum is still in rank order
        float v = 0.f;
#pragma unroll 1
        for (int r0 = 0; r0 < KS; r0 += 4) {
            float part[4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                part[r] = r0 + r < KS ? ptx::ld_cluster_f32(ptx::mapa(a, (uint32_t)(r0 + r))) : 0.f;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (r0 + r < KS) v += part[r];
        }
        const int n = n0 + nl;
        if (MODE == ABSORB || MODE == ABSORBC) {
            out[((size_t)n * g.n_h + h0) * g.width + mt * BM + tid] = __float2bfloat16_rn(v);
        } else if (MODE == OUT || MODE == OPROJ) {  // OPROJ: n_h = 1, d_h = d_model
            out[(size_t)n * g.n_h * g.d_h + (size_t)h0 * g.d_h + mt * BM + tid] = __float2bfloat16_rn(v);
        } else if (!rope_tile) {
            // latent columns: 16-byte stores of 8 columns (the row offset is per token, warp-uniform)
            const int ro = rowoff[nl];
            if (g.kv_format != KV_PLAIN)
                mx_append_block(g, ro, mt * BM + (tid & ~31), v, tid & 31);
            else
                store_cols8(out + (size_t)(ro < 0 ? 0 : ro) * g.width + mt * BM + tid, v, tid & 31, ro >= 0);
        } else if (g.kv_format != KV_PLAIN) {
            // RoPE columns into an MX cache: every lane rotates its own element of the pair
            // (2i, 2i+1) held by lanes tid, tid + 1; whole warps below d_r (a multiple of 32)
            const float w = __shfl_xor_sync(0xffffffffu, v, 1);
            if (tid < g.d_r) {
                const int i = tid >> 1;
                float cs, sn;
                rope_cos_sin(__ldg(g.pos + n), g.rf.theta[i], &cs, &sn);
                const float r = (tid & 1) ? w * sn + v * cs : v * cs - w * sn;
                mx_append_block(g, rowoff[nl], g.d_c + (tid & ~31), r, tid & 31);
            }
        } else {
            // the pair (2i, 2i+1) sits in lanes tid, tid + 1 of one warp
            const float w = __shfl_xor_sync(0xffffffffu, v, 1);
            if ((tid & 1) == 0 && tid < g.d_r && rowoff[nl] >= 0) {
                const int i = tid >> 1;
                float cs, sn;
                rope_cos_sin(__ldg(g.pos + n), g.rf.theta[i], &cs, &sn);
                *reinterpret_cast<__nv_bfloat162*>(out + (size_t)rowoff[nl] * g.width + g.d_c + 2 * i) =
                    __floats2bfloat162_rn(v * cs - w * sn, v * sn + w * cs);
            }
        }
    }
}

// grid: (m-tiles * ksplit, ceil(n_h / hpc), n-tiles), clusters of ksplit CTAs along x: the CTAs
// of a cluster share an output tile and each sums its own K range; with ksplit > 1 they add
// their partial sums through distributed shared memory and each stores a slice of the tile's
// tokens.  tmA2 is W_KR in APPEND mode (its m-tile is the last one), otherwise unused.
template <int MODE>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const GemmArgs g) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = ptx::smem_u32(smem);
    if (base & 1023u) {
        if (threadIdx.x == 0) set_device_error(MLA_ERR_UNSUPPORTED);
        return;
    }
    // the next kernel (the attention, or this GEMM's successor) may be placed as SMs free up;
    // it waits for this grid before it reads what this grid writes
    launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KS = g.ksplit, ks = (int)blockIdx.x % KS, mt = (int)blockIdx.x / KS;
    const int h0 = blockIdx.y * g.hpc, n0 = blockIdx.z * g.n_tile;
    const int kc0 = ks * g.k_chunks / KS, kper = (ks + 1) * g.k_chunks / KS - kc0;  // this CTA's K range
    const int nh = min(g.hpc, g.n_h - h0);
    const int S = g.stages, SB = stage_bytes(g.n_pad);
    const uint32_t acc_cols = tmem_cols(g.n_pad);                  // columns per head accumulator
    const uint32_t ncols = tmem_cols((int)acc_cols * g.hpc);
    const uint32_t bar_full = base + S * SB, bar_empty = bar_full + 8 * S, bar_done = bar_empty + 8 * S;
    const uint32_t slot = bar_done + 8;
    int* rowoff = reinterpret_cast<int*>(smem + (bar_done - base) + 16);  // APPEND: [n_pad] (in units of W)
    const bool a_mn = MODE != ABSORB;
    const bool rope_tile = MODE == APPEND && mt * BM >= g.d_c;
    const int total = nh * kper;                                   // chunks of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(bar_full + 8 * s, 1);
            ptx::mbar_init(bar_empty + 8 * s, 1);
        }
        ptx::mbar_init(bar_done, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(rope_tile ? &tmA2 : &tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(slot, ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<uint32_t*>(smem + (slot - base));

    if (warp == 0 && lane == 0) {
        const uint32_t bytes = (uint32_t)(A_BYTES + g.n_pad * BK * 2);
        auto load_a = [&](int c, uint32_t st, uint32_t fb) {
            const int h = h0 + chunk_head<MODE>(c, nh, kper), kc = kc0 + chunk_k<MODE>(c, nh, kper);
            if (MODE == ABSORB) {
                // W_UK rows [mt*128, +128) x cols h*d_h + kc*64 .. +64 (K-major box 64 x 128)
                ptx::tma_load_2d(st, &tmA, h * g.d_h + kc * BK, mt * BM, fb);
            } else if (MODE == APPEND || MODE == OPROJ) {
                // W_DKV / W_O (or, for the append's last tile, W_KR) rows k in [kc*64, +64) x
                // output columns m .. m + 128 (MN-major, two boxes; columns past d_r read as zeros)
                const CUtensorMap* t = rope_tile ? &tmA2 : &tmA;
                const int m0 = rope_tile ? 0 : mt * BM;
                ptx::tma_load_2d(st, t, m0, kc * BK, fb);
                ptx::tma_load_2d(st + BK * 128, t, m0 + 64, kc * BK, fb);
            } else {
                // W_UV rows c in [kc*64, +64) x cols h*d_h + mt*128 + {0, 64} (MN-major, two boxes);
                // ABSORBC: W_UQK rows k x cols h*d_c + ... (d_h holds d_c in that mode)
                ptx::tma_load_2d(st, &tmA, h * g.d_h + mt * BM, kc * BK, fb);
                ptx::tma_load_2d(st + BK * 128, &tmA, h * g.d_h + mt * BM + 64, kc * BK, fb);
            }
        };
        auto load_b = [&](int c, uint32_t st, uint32_t fb) {
            const int h = h0 + chunk_head<MODE>(c, nh, kper), kc = kc0 + chunk_k<MODE>(c, nh, kper);
            // q_nope viewed [n, n_h*d_h] (ABSORB), o_lat viewed [n, n_h*d_c] (OUT); x [n, d_model]
            // (APPEND, OPROJ) and c_q [n, d_cq] (ABSORBC) are shared by every head
            const int col = (MODE == ABSORB ? h * g.d_h : MODE == OUT ? h * g.d_c : 0) + kc * BK;
            ptx::tma_load_2d(st + A_BYTES, &tmB, col, n0, fb);
        };
        // the first ring's worth of weights goes out before the previous kernel has finished
        const int pre = total < S ? total : S;
        for (int c = 0; c < pre; ++c) {
            ptx::mbar_arrive_expect_tx(bar_full + 8 * c, bytes);
            load_a(c, base + c * SB, bar_full + 8 * c);
        }
        grid_dependency_wait();
        for (int c = 0; c < pre; ++c) load_b(c, base + c * SB, bar_full + 8 * c);
        int issued = pre;
        for (int c = pre; c < total; ++c) {
            const int s = c % S;
            if (!gwait(bar_empty + 8 * s, ((c / S) & 1u) ^ 1u, g.wait_ns)) break;
            const uint32_t st = base + s * SB, fb = bar_full + 8 * s;
            ptx::mbar_arrive_expect_tx(fb, bytes);
            load_a(c, st, fb);
            load_b(c, st, fb);
            issued = c + 1;
        }
        // the last ring's worth of loads has landed before the CTA may leave (the consumer may have
        // stopped early on a timeout); a fixed 20 ms bound
        for (int c = issued > S ? issued - S : 0; c < issued; ++c) gwait(bar_full + 8 * (c % S), (c / S) & 1u, 20000000ull);
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = ptx::idesc_bf16(BM, g.n_pad, a_mn, false);
        for (int c = 0; c < total; ++c) {
            const int s = c % S, kc = chunk_k<MODE>(c, nh, kper);
            if (!gwait(bar_full + 8 * s, (c / S) & 1u, g.wait_ns)) break;
            ptx::tc_fence_after();
            const uint32_t st = base + s * SB;
            const uint32_t d = tmem + (uint32_t)chunk_head<MODE>(c, nh, kper) * acc_cols;
            const uint64_t da = a_mn ? ptx::desc_sw128(st, BK * 128, 1024) : ptx::desc_sw128(st, 16, 1024);
            const uint64_t db = ptx::desc_sw128(st + A_BYTES, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // K-major A: +32 B per 16-wide K step; MN-major A: +16 rows of 128 B
                const uint64_t a_off = a_mn ? (uint64_t)((kk * 2048) >> 4) : (uint64_t)((kk * 32) >> 4);
                ptx::mma_ss(d, da + a_off, db + (uint64_t)((kk * 32) >> 4), idesc, (kc | kk) ? 1u : 0u);
            }
            ptx::tc_commit(bar_empty + 8 * s);
        }
        ptx::tc_commit(bar_done);
    } else if (warp >= 2) {
        const int qd = warp & 3;
        const int row = qd * 32 + lane;  // m within the tile
        if ((MODE == ABSORB || MODE == ABSORBC) && g.q_rope) {
            grid_dependency_wait();  // q_rope and pos come from earlier kernels
            absorb_rope(g, n0, threadIdx.x - 64);
        }
        const int tid = threadIdx.x - 64, n_here = min(g.n_pad, g.n_tokens - n0);
        if (MODE == APPEND) {
            // where each token of the tile goes (inputs of earlier kernels: after the wait)
            grid_dependency_wait();
            for (int i = tid; i < n_here; i += NTHREADS - 64) {
                const long long r = append_row(g, n0 + i);
                rowoff[i] = r < 0 ? -1 : (int)(r / g.width);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        // the four epilogue warps agree on the outcome of the wait (they meet at named barriers)
        bool done_ok = false;
        if (MODE == APPEND || KS > 1) {
            const bool mine = gwait(bar_done, 0, g.wait_ns);
            uint32_t all;
            asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\t"
                         "selp.u32 %0, 1, 0, q;\n\t}"
                         : "=r"(all)
                         : "r"((uint32_t)mine)
                         : "memory");
            done_ok = all != 0;
        }
        if (KS > 1) {
            // this CTA's partial sums, [n_pad][128] fp32, into the ring (idle: every MMA is done)
            if (done_ok) {
                ptx::tc_fence_after();
                float* stg = reinterpret_cast<float*>(smem);
                const uint32_t taddr = tmem + ((uint32_t)(qd * 32) << 16);
                for (int c0 = 0; c0 < g.n_pad; c0 += 32) {
                    uint32_t r[32];
                    ptx::tmem_ld32(taddr + c0, r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c0 + i < g.n_pad) stg[(c0 + i) * BM + row] = __uint_as_float(r[i]);
                }
            }
        } else if (MODE == APPEND && done_ok) {
            ptx::tc_fence_after();
            bf16* pool = reinterpret_cast<bf16*>(g.pool);
            const uint32_t taddr = tmem + ((uint32_t)(qd * 32) << 16);
            if (!rope_tile) {
                // latent columns: per token, the 128 threads hold 128 consecutive values, stored
                // 8 columns per 16-byte store (MX cache: one 32-column block per warp)
                const int c = mt * BM + row;
                for (int c0 = 0; c0 < g.n_pad; c0 += 32) {
                    uint32_t r[32];
                    ptx::tmem_ld32(taddr + c0, r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (c0 + i >= n_here) break;  // warp-uniform
                        const int ro = rowoff[c0 + i];
                        if (g.kv_format != KV_PLAIN)
                            mx_append_block(g, ro, c - lane, __uint_as_float(r[i]), lane);
                        else
                            store_cols8(pool + (size_t)(ro < 0 ? 0 : ro) * g.width + c, __uint_as_float(r[i]), lane,
                                        ro >= 0);
                    }
                }
            } else {
                // RoPE columns: the pair (2i, 2i+1) sits in two threads, so the fp32 values go
                // through shared memory (the ring is idle now: every MMA has completed)
                float* stg = reinterpret_cast<float*>(smem);  // [n_pad][d_r]
                for (int c0 = 0; c0 < g.n_pad; c0 += 32) {
                    uint32_t r[32];
                    ptx::tmem_ld32(taddr + c0, r);
                    ptx::tmem_wait_ld();
                    if (row < g.d_r) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c0 + i < g.n_pad) stg[(c0 + i) * g.d_r + row] = __uint_as_float(r[i]);
                    }
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (g.kv_format != KV_PLAIN) {
                    // MX cache: warp w codes blocks (token, b) = items w, w + 4, ...; lane l
                    // rotates element 32 b + l of the token's RoPE key
                    const int nb = g.d_r / MX_BLOCK;
                    for (int e = tid >> 5; e < n_here * nb; e += (NTHREADS - 64) / 32) {
                        const int nl = e / nb, col = (e % nb) * MX_BLOCK + lane, i = col >> 1;
                        float cs, sn;
                        rope_cos_sin(__ldg(g.pos + n0 + nl), g.rf.theta[i], &cs, &sn);
                        const float x0 = stg[nl * g.d_r + 2 * i], x1 = stg[nl * g.d_r + 2 * i + 1];
                        const float v = (col & 1) ? x0 * sn + x1 * cs : x0 * cs - x1 * sn;
                        mx_append_block(g, rowoff[nl], g.d_c + col - lane, v, lane);
                    }
                }
                const int half = g.kv_format != KV_PLAIN ? 0 : g.d_r / 2;
                for (int e = tid; e < n_here * half; e += NTHREADS - 64) {
                    const int nl = e / half, i = e % half;
                    if (rowoff[nl] < 0) continue;
                    float cs, sn;
                    rope_cos_sin(__ldg(g.pos + n0 + nl), g.rf.theta[i], &cs, &sn);
                    const float x0 = stg[nl * g.d_r + 2 * i], x1 = stg[nl * g.d_r + 2 * i + 1];
                    *reinterpret_cast<__nv_bfloat162*>(pool + (size_t)rowoff[nl] * g.width + g.d_c + 2 * i) =
                        __floats2bfloat162_rn(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
                }
            }
        } else if (MODE != APPEND && gwait(bar_done, 0, g.wait_ns)) {
            ptx::tc_fence_after();
            bf16* out = reinterpret_cast<bf16*>(g.out);
            for (int j = 0; j < nh; ++j) {
                const int h = h0 + j;
                const uint32_t taddr = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)j * acc_cols;
                for (int c0 = 0; c0 < g.n_pad; c0 += 32) {  // reads stay inside the allocation (>= 32 columns)
                    uint32_t r[32];
                    ptx::tmem_ld32(taddr + c0, r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int n = n0 + c0 + i;
                        if (c0 + i < g.n_pad && n < g.n_tokens) {
                            const bf16 v = __float2bfloat16_rn(__uint_as_float(r[i]));
                            if (MODE == ABSORB || MODE == ABSORBC)
                                out[((size_t)n * g.n_h + h) * g.width + mt * BM + row] = v;
                            else
                                out[(size_t)n * g.n_h * g.d_h + (size_t)h * g.d_h + mt * BM + row] = v;
                        }
                    }
                }
            }
        }
    }
    if (KS > 1) {
        // every thread of the cluster passes both barriers, whatever its waits returned
        __syncwarp();
        ptx::cluster_sync();  // all partial sums are staged
        if (warp >= 2) split_store<MODE>(g, base, rowoff, mt, h0, n0, ks, rope_tile, threadIdx.x - 64);
        __syncwarp();
        ptx::cluster_sync();  // the peers have finished reading this CTA's shared memory
    }
    // every MMA issued completes before TMEM is freed (the epilogue's own wait may have run out):
    // the issuing thread waits for its final commit with a fixed 20 ms bound
    if (warp == 1 && lane == 0) gwait(bar_done, 0, 20000000ull);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, ncols);
    }
}

// 2-D bf16 map: inner extent `inner` elements with row pitch `pitch_elems`, `rows` rows, box
// (64, box_rows), 128-byte swizzle; reads past the extents return zeros.
inline bool encode_2d(CUtensorMap* tm, const void* p, uint64_t inner, uint64_t rows, uint64_t pitch_elems,
                      uint32_t box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) !=
                cudaSuccess ||
            r != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
    }
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {pitch_elems * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int n_pad_for(int n) {
    int p = n < MAX_N ? n : MAX_N;
    return (p + 15) & ~15;
}

inline mla_status launch(const GemmArgs& g0, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a2,
                         int m_tiles, int n_h, const Tuning& t, cudaStream_t stream) {
    GemmArgs g = g0;
    g.wait_ns = t.wait_ns;
    if (g.n_tile == 0) g.n_tile = MAX_N;
    g.hpc = 1;
    if (t.hpc > 0) g.hpc = t.hpc < max_heads_per_cta(g.n_pad) ? t.hpc : max_heads_per_cta(g.n_pad);
    // K split over a cluster by default when a deep K (d_model or n_h*d_h, streamed per CTA)
    // would otherwise leave most SMs idle
    const bool deep_k = g.mode == APPEND || g.mode == OPROJ;
    const long long ctas = (long long)m_tiles * ((g.n_tokens + g.n_tile - 1) / g.n_tile);
    int ksp = t.ksplit > 0 ? t.ksplit : (deep_k && ctas < SPLIT_BELOW_CTAS ? MAX_KSPLIT : 1);
    if (ksp > MAX_KSPLIT) ksp = MAX_KSPLIT;
    if (ksp > g.k_chunks) ksp = g.k_chunks;
    if (g.hpc != 1 || ksp < 1) ksp = 1;
    g.ksplit = ksp;
    // ring depth: APPEND and OPROJ without a split stream a deep K per CTA, as deep a ring as fits;
    // never deeper than the chunks one CTA streams; with a split, deep enough to stage the
    // partial sums ([n_pad][128] fp32) where the ring was
    const int chunks = g.hpc * ((g.k_chunks + ksp - 1) / ksp), mx = max_stages(g.n_pad);
    int S = ksp > 1 ? SPLIT_STAGES : deep_k ? mx : stages_for(g.n_pad);
    if (t.stages > 0) S = t.stages;
    if (S > chunks) S = chunks;
    if (ksp > 1) {
        const int need = (g.n_pad * BM * 4 + stage_bytes(g.n_pad) - 1) / stage_bytes(g.n_pad);
        if (S < need) S = need;
    }
    if (S > mx) S = mx;
    if (S < 1 || (ksp > 1 && S * stage_bytes(g.n_pad) < g.n_pad * BM * 4)) return MLA_ERR_UNSUPPORTED;
    g.stages = S;
    const int smem = smem_bytes(g.n_pad, g.stages);
    // one instantiation per mode: each launch fetches only its own code (cold after every L2
    // flush; instruction fetch stalls dominated this short kernel when the modes shared one)
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, GemmArgs) =
        g.mode == ABSORB ? tc_gemm_kernel<ABSORB>
        : g.mode == OUT  ? tc_gemm_kernel<OUT>
        : g.mode == OPROJ ? tc_gemm_kernel<OPROJ>
        : g.mode == ABSORBC ? tc_gemm_kernel<ABSORBC>
                          : tc_gemm_kernel<APPEND>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return MLA_ERR_CUDA;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(m_tiles * ksp, (n_h + g.hpc - 1) / g.hpc, (g.n_tokens + g.n_tile - 1) / g.n_tile);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (t.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (ksp > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)ksp;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    lc.attrs = attr;
    lc.numAttrs = na;
    if (cudaLaunchKernelEx(&lc, kern, a, b, a2, g) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

}  // namespace tcg

inline bool tc_gemm_absorb_supported(const mla_config* c, int n, int cc_major, int cc_minor) {
    return c->dtype == MLA_BF16 && cc_major == 10 && cc_minor == 3 && n > 0 && c->d_nope % 64 == 0 &&
           c->d_latent % 128 == 0 && ((long long)c->n_heads * c->d_nope) % 8 == 0;
}
inline bool tc_gemm_out_supported(const mla_config* c, int n, int cc_major, int cc_minor) {
    return c->dtype == MLA_BF16 && cc_major == 10 && cc_minor == 3 && n > 0 && c->d_nope % 128 == 0 &&
           c->d_latent % 64 == 0;
}

// the whole of q_cat for mla_absorb_q: the GEMM half and, in the first m-tile's CTAs, RoPE
inline mla_status tc_gemm_absorb(const mla_config* c, const void* q_nope, const void* q_rope, const int* pos,
                                 const void* w_uk, void* q_cat, int n, const tcg::Tuning& t, cudaStream_t stream) {
    tcg::GemmArgs g{};
    g.mode = tcg::ABSORB;
    g.n_tokens = n;
    g.q_rope = reinterpret_cast<const bf16*>(q_rope);
    g.pos = pos;
    g.d_r = c->d_rope;
    rope_freq_fill(&g.rf, c->d_rope, c->rope_base);
    g.n_pad = tcg::n_pad_for(n);
    g.k_chunks = c->d_nope / tcg::BK;
    g.n_h = c->n_heads; g.d_h = c->d_nope; g.d_c = c->d_latent; g.width = c->d_latent + c->d_rope;
    g.out = q_cat;
    const uint64_t hd = (uint64_t)c->n_heads * c->d_nope;
    CUtensorMap ta, tb;
    if (!tcg::encode_2d(&ta, w_uk, hd, (uint64_t)c->d_latent, hd, tcg::BM) ||
        !tcg::encode_2d(&tb, q_nope, hd, (uint64_t)n, hd, (uint32_t)g.n_pad))
        return MLA_ERR_CUDA;
    return tcg::launch(g, ta, tb, ta, c->d_latent / tcg::BM, c->n_heads, t, stream);
}

inline mla_status tc_gemm_out(const mla_config* c, const void* o_lat, const void* w_uv, void* o, int n,
                              const tcg::Tuning& t, cudaStream_t stream) {
    tcg::GemmArgs g{};
    g.mode = tcg::OUT;
    g.n_tokens = n;
    g.n_pad = tcg::n_pad_for(n);
    g.k_chunks = c->d_latent / tcg::BK;
    g.n_h = c->n_heads; g.d_h = c->d_nope; g.d_c = c->d_latent; g.width = c->d_latent + c->d_rope;
    g.out = o;
    const uint64_t hd = (uint64_t)c->n_heads * c->d_nope, hc = (uint64_t)c->n_heads * c->d_latent;
    CUtensorMap ta, tb;
    if (!tcg::encode_2d(&ta, w_uv, hd, (uint64_t)c->d_latent, hd, 64) ||
        !tcg::encode_2d(&tb, o_lat, hc, (uint64_t)n, hc, (uint32_t)g.n_pad))
        return MLA_ERR_CUDA;
    return tcg::launch(g, ta, tb, ta, c->d_nope / tcg::BM, c->n_heads, t, stream);
}

inline bool tc_gemm_absorbc_supported(const mla_config* c, int d_cq, int n, int cc_major, int cc_minor) {
    return c->dtype == MLA_BF16 && cc_major == 10 && cc_minor == 3 && n > 0 && d_cq % 64 == 0 &&
           c->d_latent % 128 == 0 && c->d_rope % 2 == 0 && (c->d_rope * 2) % 16 == 0;
}

// The absorbed query from the compressed query latent: one CTA per (128 latent columns, head,
// token tile), W_UQK's head slab as the MN-major A operand (the OUT mode's addressing with
// d_h := d_c), c_q as B for every head, the ABSORB mode's epilogue and RoPE half.
inline mla_status tc_gemm_absorb_compressed(const mla_config* c, int d_cq, const void* c_q, const void* q_rope,
                                            const int* pos, const void* w_uqk, void* q_cat, int n,
                                            const tcg::Tuning& t, cudaStream_t stream) {
    tcg::GemmArgs g{};
    g.mode = tcg::ABSORBC;
    g.n_tokens = n;
    g.q_rope = reinterpret_cast<const bf16*>(q_rope);
    g.pos = pos;
    g.d_r = c->d_rope;
    rope_freq_fill(&g.rf, c->d_rope, c->rope_base);
    g.n_pad = tcg::n_pad_for(n);
    g.k_chunks = d_cq / tcg::BK;
    g.n_h = c->n_heads; g.d_h = c->d_latent; g.d_c = c->d_latent; g.width = c->d_latent + c->d_rope;
    g.out = q_cat;
    const uint64_t hc = (uint64_t)c->n_heads * c->d_latent;
    CUtensorMap ta, tb;
    if (!tcg::encode_2d(&ta, w_uqk, hc, (uint64_t)d_cq, hc, 64) ||
        !tcg::encode_2d(&tb, c_q, (uint64_t)d_cq, (uint64_t)n, (uint64_t)d_cq, (uint32_t)g.n_pad))
        return MLA_ERR_CUDA;
    return tcg::launch(g, ta, tb, ta, c->d_latent / tcg::BM, c->n_heads, t, stream);
}

// a dense projection out[n, :] = in[n, :] . W with W [K, M] row-major (M contiguous), the
// OPROJ mode: W as the MN-major A operand, K a multiple of 64, M of 128, bf16
inline bool tc_gemm_dense_supported(const mla_config* c, long long K, long long M, int n, int cc_major,
                                    int cc_minor) {
    return c->dtype == MLA_BF16 && cc_major == 10 && cc_minor == 3 && n > 0 && K % 64 == 0 && M % 128 == 0 &&
           K <= (1LL << 24) && M <= (1LL << 24);
}

// One CTA per (128 output columns, token tile).  W (168 MB for W_O, W_Q at DeepSeek-V2 sizes)
// can be larger than L2, so up to 256 tokens share one token tile and W is streamed once; K is
// then split over clusters of 8 CTAs when the output tiles alone would leave SMs idle.
inline mla_status tc_gemm_dense(const mla_config* c, const void* in, const void* w, void* out, long long K,
                                long long M, int n, const tcg::Tuning& t, cudaStream_t stream,
                                long long in_pitch = 0) {  // elements per input row (0: K)
    tcg::GemmArgs g{};
    g.mode = tcg::OPROJ;
    g.n_tokens = n;
    g.n_pad = tcg::n_pad_for(n);
    g.n_tile = n <= tcg::MAX_N ? g.n_pad : tcg::MAX_N;
    g.k_chunks = (int)(K / tcg::BK);
    g.n_h = 1;
    g.d_h = (int)M;  // the epilogue's output row pitch
    g.out = out;
    CUtensorMap ta, tb;
    if (!tcg::encode_2d(&ta, w, (uint64_t)M, (uint64_t)K, (uint64_t)M, 64) ||
        !tcg::encode_2d(&tb, in, (uint64_t)K, (uint64_t)n, (uint64_t)(in_pitch > 0 ? in_pitch : K), (uint32_t)g.n_pad))
        return MLA_ERR_CUDA;
    return tcg::launch(g, ta, tb, ta, (int)(M / tcg::BM), 1, t, stream);
}

inline bool tc_gemm_append_supported(const mla_config* c, int n, int cc_major, int cc_minor) {
    return c->dtype == MLA_BF16 && cc_major == 10 && cc_minor == 3 && n > 0 && c->d_model % 64 == 0 &&
           c->d_latent % 128 == 0 && c->d_rope > 0 && c->d_rope <= 128 && (c->d_rope * 2) % 16 == 0;
}

// mla_cache_append on the tensor cores: one CTA per (128 output columns, token tile); the
// last column tile is W_KR, rotated and stored through shared memory.  Few tokens (decode
// steps) use 32-token tiles and split K over clusters of 8 CTAs, so that many CTAs share the
// weight stream.
inline mla_status tc_gemm_append(const mla_config* c, const mla_cache* k, const void* x, const void* w_dkv,
                                 const void* w_kr, const int32_t* seq_idx, const int32_t* pos, int n,
                                 const tcg::Tuning& t, cudaStream_t stream) {
    tcg::GemmArgs g{};
    g.mode = tcg::APPEND;
    g.n_tokens = n;
    g.n_tile = n <= 512 ? 32 : tcg::MAX_N;
    g.n_pad = tcg::n_pad_for(n < g.n_tile ? n : g.n_tile);
    g.k_chunks = c->d_model / tcg::BK;
    g.n_h = 1;
    g.d_c = c->d_latent;
    g.d_r = c->d_rope;
    g.width = c->d_latent + c->d_rope;
    g.pos = pos;
    rope_freq_fill(&g.rf, c->d_rope, c->rope_base);
    g.pool = k->pool;
    g.page_table = k->page_table;
    g.seq_idx = seq_idx;
    g.max_pages = k->max_pages;
    g.batch = k->batch;
    g.page_size = c->page_size;
    g.num_pages = k->num_pages;
    g.kv_format = k->kv_format;
    g.scales = k->kv_scales;
    CUtensorMap ta, ta2, tb;
    if (!tcg::encode_2d(&ta, w_dkv, (uint64_t)c->d_latent, (uint64_t)c->d_model, (uint64_t)c->d_latent, 64) ||
        !tcg::encode_2d(&ta2, w_kr, (uint64_t)c->d_rope, (uint64_t)c->d_model, (uint64_t)c->d_rope, 64) ||
        !tcg::encode_2d(&tb, x, (uint64_t)c->d_model, (uint64_t)n, (uint64_t)c->d_model, (uint32_t)g.n_pad))
        return MLA_ERR_CUDA;
    return tcg::launch(g, ta, tb, ta2, c->d_latent / tcg::BM + 1, 1, t, stream);
}

}  // namespace mla
