// Un-absorbed causal prefill (sm_103a): the chain of the operator-notes page, section 2
// ("Restore K, V from c_kv", then "Standard scaled-dot-product attention"), with the decoupled
// RoPE key of the MLA glossary.  For a prefill of T queries over L = q_start + T cached tokens
// this form costs 2 L d_c n_h d_h * 2 (restoring K and V) plus about T^2 n_h (d_h + d_r + d_h)
// FLOPs, against T^2 n_h (2 d_c + d_r) for the absorbed form: 3.0 against 9.35 TFLOP at T=8192.
//
// Three steps, all on the device:
//   1. prep_kernel gathers the sequence's cache rows [L, d_c + d_r] into one contiguous buffer
//      and builds the un-absorbed query qu[h][t] = [q_nope[t, h] | RoPE(q_rope[t, h], q_start+t)]
//      (head-major, so that one head's query tile is a plain 2-D box);
//   2. two dense tcgen05 GEMMs restore K = c_kv . W_UK and V = c_kv . W_UV ([L, n_h d_h] each);
//   3. flash_kernel: causal attention per (head, 128-query tile) with 192-wide scores
//      s = [q_nope | q_rope] . [K_h | k_rope] * scale and 128-wide values V_h.
//
// flash_kernel, one CTA per (head, query tile), 192 threads:
//   warp 0      TMA: the query tile once (three 64-column boxes), then per 128-key tile the key
//               tile (K_h two boxes, k_rope one box) and V_h (two boxes) into a 2-stage ring;
//   warp 1      MMA issue: S_j = Q . K_j^T (12 MMAs, M=128, N=128, K=16, both operands in shared
//               memory) into one of two TMEM score buffers, then O += P_{j-1} . V_{j-1}
//               (8 MMAs, N=128, P from TMEM);
//   warps 2-5   softmax, one query row per thread (the TMEM lane): scale, causal mask, running
//               max raised lazily (only when it grows by more than 2^8, as in the decode kernel),
//               P to TMEM as bf16 pairs, O rescaled in TMEM when the max moved; the epilogue
//               writes o[t, h d_h : (h+1) d_h] and lse.
// TMEM: S double buffer [0,256), O [256,384), P double buffer [384,512).  Every wait is bounded.
#pragma once

#include <cudaTypedefs.h>

#include "mla_common.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tcf {

constexpr int DH = 128, DR = 64, DQ = DH + DR;      // value width, RoPE width, score width
constexpr int BQ = 128, BKEY = 128;                // query and key tile
constexpr int QCH = DQ / 64;                       // 64-column chunks of a query / key row: 3
constexpr int Q_BYTES = QCH * BQ * 128;            // 48 KB
constexpr int K_BYTES = QCH * BKEY * 128;          // 48 KB
constexpr int V_BYTES = (DH / 64) * BKEY * 128;    // 32 KB
constexpr int KV_STAGE = K_BYTES + V_BYTES;        // 80 KB
constexpr int KV_STAGES = 2;
constexpr int OFF_KV = Q_BYTES;
enum {
    F_QFULL = 0,
    F_KVFULL = 1,                 // [2]
    F_KVEMPTY = F_KVFULL + 2,     // [2]
    F_SFULL = F_KVEMPTY + 2,      // [2]
    F_SFREE = F_SFULL + 2,        // [2] four softmax warps
    F_PFULL = F_SFREE + 2,        // [2] four softmax warps
    F_PVDONE = F_PFULL + 2,       // [2]
    F_DONE = F_PVDONE + 2,
    F_NBARS
};
constexpr int OFF_BARS = OFF_KV + KV_STAGES * KV_STAGE;
constexpr int OFF_MISC = OFF_BARS + F_NBARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr int NTHREADS = 192;
constexpr uint32_t TM_S = 0, TM_O = 256, TM_P = 384;
constexpr float TAU = 8.0f;
constexpr float LN2 = 0.6931471805599453f;
constexpr uint32_t IDESC_S = ptx::idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_O = ptx::idesc_bf16(128, 128, false, true);

struct PrepArgs {
    const bf16* pool;          // [num_pages, P, W]
    const int* page_row;       // the sequence's page table row
    int max_pages;
    long long num_pages;
    int page_size, width;      // P, W = d_c + d_r
    int n_keys;                // L
    bf16* rows;                // out: [L, W]
    const bf16* q_nope;        // [T, n_h, d_h]
    const bf16* q_rope;        // [T, n_h, d_r], not rotated
    int n_queries, n_h, q_start;
    RopeFreq rf;
    bf16* qu;                  // out: [n_h, T, d_h + d_r]
};

// One 16-byte group per item: first the L * W / 8 row groups, then the T * n_h * (d_h + d_r) / 8
// query groups (a RoPE group rotates its four pairs).
__global__ void __launch_bounds__(256) prep_kernel(PrepArgs p) {
    launch_dependents();
    grid_dependency_wait();  // the cache rows and the queries come from earlier kernels
    const long long row_groups = (long long)p.n_keys * (p.width / 8);
    const int qg = (DH + DR) / 8;
    const long long q_groups = (long long)p.n_queries * p.n_h * qg;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < row_groups + q_groups;
         i += (long long)gridDim.x * blockDim.x) {
        if (i < row_groups) {
            const long long t = i / (p.width / 8);
            const int c8 = (int)(i % (p.width / 8));
            int page = __ldg(p.page_row + t / p.page_size);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (page >= 0 && page < p.num_pages) {
                v = *reinterpret_cast<const uint4*>(p.pool + ((long long)page * p.page_size + t % p.page_size) * p.width +
                                                    8 * c8);
            } else if (c8 == 0) {
                set_device_error(MLA_ERR_DEVICE_BOUNDS);
            }
            *reinterpret_cast<uint4*>(p.rows + t * p.width + 8 * c8) = v;
        } else {
            const long long j = i - row_groups;
            const int g = (int)(j % qg);
            const long long th = j / qg;          // t * n_h + h
            const long long t = th / p.n_h;
            const int h = (int)(th % p.n_h);
            uint4 v;
            if (g < DH / 8) {
                v = *reinterpret_cast<const uint4*>(p.q_nope + th * DH + 8 * g);
            } else {
                const int c0 = 8 * (g - DH / 8);  // first RoPE column of the group
                const uint4 raw = *reinterpret_cast<const uint4*>(p.q_rope + th * DR + c0);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
                    const float x0 = __bfloat162float(pr.x), x1 = __bfloat162float(pr.y);
                    float cs, sn;
                    rope_cos_sin(p.q_start + (int)t, p.rf.theta[c0 / 2 + k], &cs, &sn);
                    const __nv_bfloat162 r = __floats2bfloat162_rn(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
                    o[k] = *reinterpret_cast<const uint32_t*>(&r);
                }
                v = make_uint4(o[0], o[1], o[2], o[3]);
            }
            *reinterpret_cast<uint4*>(p.qu + ((long long)h * p.n_queries + t) * (DH + DR) + 8 * g) = v;
        }
    }
}

struct FlashArgs {
    int n_queries, n_keys, n_h, q_start;
    int rope_col;              // first RoPE column of a gathered cache row (d_c)
    float scale_log2;
    bf16* o;                   // [T, n_h * d_h]
    float* lse;                // [T, n_h]
    unsigned long long wait_ns;
};

struct FWait {
    unsigned long long limit_ns;
    volatile int* abort;
    bool ignore_abort;
};

__device__ __forceinline__ bool fwait(uint32_t bar, uint32_t parity, const FWait& w) {
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (i & 1u) {
            if (!w.ignore_abort && *w.abort) return false;
            const unsigned long long t = globaltimer_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > w.limit_ns) {
                *w.abort = 1;
                set_device_error(MLA_ERR_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool fwait_warp(uint32_t bar, uint32_t parity, const FWait& w, int lane) {
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const bool ok = ptx::mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if (i & 1u) {
            int stop = 0;
            if (lane == 0) {
                if (*w.abort) stop = 1;
                const unsigned long long t = globaltimer_ns();
                if (t0 == 0) t0 = t;
                else if (t - t0 > w.limit_ns) {
                    *w.abort = 1;
                    set_device_error(MLA_ERR_DEVICE_TIMEOUT);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        }
    }
}

__device__ __forceinline__ uint32_t fbar(uint32_t base, int i) { return base + OFF_BARS + 8u * (uint32_t)i; }

// key tiles that query tile qt sees: keys [0, q_start + q0 + BQ) within [0, L)
__device__ __forceinline__ int key_tiles(const FlashArgs& a, int q0) {
    long long hi = (long long)a.q_start + q0 + BQ;
    if (hi > a.n_keys) hi = a.n_keys;
    return (int)((hi + BKEY - 1) / BKEY);
}

// ----------------------------------------------------------------------------- warp 0: TMA
__device__ __forceinline__ void f_producer(const FlashArgs& a, const CUtensorMap* tmq, const CUtensorMap* tmk,
                                           const CUtensorMap* tmr, const CUtensorMap* tmv, uint32_t base, int h,
                                           int q0, int n_t, const FWait& wc) {
    grid_dependency_wait();  // prep and the restoring GEMMs wrote what this kernel reads
    const uint32_t qf = fbar(base, F_QFULL);
    ptx::mbar_arrive_expect_tx(qf, (uint32_t)Q_BYTES);
    for (int cc = 0; cc < QCH; ++cc) ptx::tma_load_2d(base + cc * BQ * 128, tmq, cc * 64, h * a.n_queries + q0, qf);
    int j = 0;
    bool ok = true;
    for (; j < n_t; ++j) {
        const int st = j & 1;
        if (j >= 2 && !fwait(fbar(base, F_KVEMPTY + st), ((j >> 1) & 1) ^ 1, wc)) { ok = false; break; }
        const uint32_t fb = fbar(base, F_KVFULL + st), dst = base + OFF_KV + st * KV_STAGE;
        const int key0 = j * BKEY;
        ptx::mbar_arrive_expect_tx(fb, (uint32_t)KV_STAGE);
        ptx::tma_load_2d(dst, tmk, h * DH, key0, fb);                       // K_h, columns 0-63
        ptx::tma_load_2d(dst + BKEY * 128, tmk, h * DH + 64, key0, fb);     // K_h, columns 64-127
        ptx::tma_load_2d(dst + 2 * BKEY * 128, tmr, a.rope_col, key0, fb);   // k_rope
        ptx::tma_load_2d(dst + K_BYTES, tmv, h * DH, key0, fb);             // V_h, columns 0-63
        ptx::tma_load_2d(dst + K_BYTES + BKEY * 128, tmv, h * DH + 64, key0, fb);
    }
    FWait w2 = wc;  // loads still in flight land before the CTA leaves (bounded)
    w2.ignore_abort = true;
    w2.limit_ns = 20000000ull;
    if (!ok) {
        for (int k = j - 2 < 0 ? 0 : j - 2; k < j; ++k) fwait(fbar(base, F_KVFULL + (k & 1)), (k >> 1) & 1, w2);
    }
    fwait(qf, 0, w2);
}

// ----------------------------------------------------------------------------- warp 1: MMA
// Run by the whole warp: every lane computes the descriptors, one elected lane issues (issuing
// from a single active lane costs issue slots that the softmax warps on the same
// sub-partitions need).
__device__ __forceinline__ void f_mma(uint32_t base, uint32_t tmem, int n_t, const FWait& wc, int lane) {
    bool ok = fwait_warp(fbar(base, F_QFULL), 0, wc, lane);
    const uint64_t qd = ptx::desc_sw128(base, 16, 1024);
    auto qk = [&](int j) -> bool {
        const int st = j & 1;
        if (!fwait_warp(fbar(base, F_KVFULL + st), (j >> 1) & 1, wc, lane)) return false;
        if (j >= 2 && !fwait_warp(fbar(base, F_SFREE + st), ((j >> 1) & 1) ^ 1, wc, lane)) return false;
        ptx::tc_fence_after();
        const uint64_t kd = ptx::desc_sw128(base + OFF_KV + st * KV_STAGE, 16, 1024);
        const uint32_t d = tmem + TM_S + st * 128;
#pragma unroll
        for (int cc = 0; cc < QCH; ++cc)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t off = (uint64_t)((cc * BQ * 128 + kk * 32) >> 4);
                ptx::mma_ss_elect(d, qd + off, kd + off, IDESC_S, (cc | kk) ? 1u : 0u);
            }
        ptx::tc_commit_elect(fbar(base, F_SFULL + st));
        return true;
    };
    auto pv = [&](int i) -> bool {
        const int st = i & 1;
        if (!fwait_warp(fbar(base, F_PFULL + st), (i >> 1) & 1, wc, lane)) return false;
        ptx::tc_fence_after();
        // V is the MN-major B operand: 64-column chunks 16 KB apart, 16 keys = 2 KB per MMA
        const uint64_t vd = ptx::desc_sw128(base + OFF_KV + st * KV_STAGE + K_BYTES, BKEY * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < BKEY / 16; ++kk)
            ptx::mma_ts_elect(tmem + TM_O, tmem + TM_P + st * 64 + kk * 8, vd + (uint64_t)((kk * 2048) >> 4), IDESC_O,
                              (i > 0 || kk > 0) ? 1u : 0u);
        ptx::tc_commit_elect(fbar(base, F_PVDONE + st));
        ptx::tc_commit_elect(fbar(base, F_KVEMPTY + st));
        return true;
    };
    for (int j = 0; ok && j < n_t; ++j) {
        ok = qk(j);
        if (ok && j >= 1) ok = pv(j - 1);
    }
    if (ok) pv(n_t - 1);
    // every MMA issued completes before TMEM is freed (a fixed 20 ms bound)
    __syncwarp();
    ptx::tc_commit_elect(fbar(base, F_DONE));
    FWait w2 = wc;
    w2.ignore_abort = true;
    w2.limit_ns = 20000000ull;
    fwait_warp(fbar(base, F_DONE), 0, w2, lane);
}

// ----------------------------------------------------------------------------- warps 2-5
__device__ __forceinline__ void f_softmax(const FlashArgs& a, uint32_t base, uint32_t tmem, int h, int q0, int n_t,
                                          int warp, int lane, const FWait& wc) {
    const int qd = warp & 3;
    const int i = qd * 32 + lane;  // query row of the tile (TMEM lane)
    const uint32_t lb = (uint32_t)(qd * 32) << 16;
    const long long qpos = (long long)a.q_start + q0 + i;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_t; ++j) {
        const int st = j & 1;
        if (!fwait_warp(fbar(base, F_SFULL + st), (j >> 1) & 1, wc, lane)) { ok = false; break; }
        ptx::tc_fence_after();
        float s[BKEY];
#pragma unroll
        for (int c4 = 0; c4 < BKEY / 32; c4 += 2) {
            uint32_t r0[32], r1[32];
            ptx::tmem_ld32(tmem + lb + TM_S + st * 128 + 32 * c4, r0);
            ptx::tmem_ld32(tmem + lb + TM_S + st * 128 + 32 * (c4 + 1), r1);
            ptx::tmem_wait_ld_regs(r0);
            ptx::tmem_wait_ld_regs(r1);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                s[32 * c4 + k] = __uint_as_float(r0[k]);
                s[32 * (c4 + 1) + k] = __uint_as_float(r1[k]);
            }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(fbar(base, F_SFREE + st));
        // keys after the query's position are masked (-inf); only the tiles on the diagonal have
        // any, so the others take the loop without the compare.  The running max m is in scaled
        // log2 units; the scale is positive, so the raw maximum scales to the scaled one, and
        // p = 2^(s * scale - m) is one FFMA and one ex2 per score.
        const long long key0 = (long long)j * BKEY;
        const int allowed = qpos - key0 + 1 > BKEY ? BKEY : (int)(qpos - key0 + 1);  // keys key0 .. qpos
        float mraw = -INFINITY;
        if (__all_sync(0xffffffffu, allowed >= BKEY)) {
#pragma unroll
            for (int c = 0; c < BKEY; ++c) mraw = fmaxf(mraw, s[c]);
        } else {
#pragma unroll
            for (int c = 0; c < BKEY; ++c) {
                s[c] = c < allowed ? s[c] : -INFINITY;
                mraw = fmaxf(mraw, s[c]);
            }
        }
        const float mx = mraw * a.scale_log2;
        float alpha = 1.f;
        if (mx > m + TAU) {
            alpha = ptx::ex2(m - mx);  // 0 while m is -inf
            m = mx;
            l *= alpha;
        }
        float sum = 0.f;
        uint32_t pk[BKEY / 2];
        const float sl = a.scale_log2, nm = -m;
#pragma unroll
        for (int c = 0; c < BKEY / 2; ++c) {
            const float p0 = ptx::ex2(fmaf(s[2 * c], sl, nm)), p1 = ptx::ex2(fmaf(s[2 * c + 1], sl, nm));
            sum += p0 + p1;
            pk[c] = ptx::pack_bf16(p0, p1);
        }
        l += sum;
        // P buffer st is free once PV(j-2) has completed
        if (j >= 2 && !fwait_warp(fbar(base, F_PVDONE + st), ((j >> 1) & 1) ^ 1, wc, lane)) { ok = false; break; }
        // O rows whose max moved are rescaled once every earlier PV has completed
        if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
            const int jp = j - 1;
            if (!fwait_warp(fbar(base, F_PVDONE + (jp & 1)), (jp >> 1) & 1, wc, lane)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll 1
            for (int c4 = 0; c4 < DH / 32; c4 += 2) {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(tmem + lb + TM_O + 32 * c4, r0);
                ptx::tmem_ld32(tmem + lb + TM_O + 32 * (c4 + 1), r1);
                ptx::tmem_wait_ld_regs(r0);
                ptx::tmem_wait_ld_regs(r1);
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    r0[k] = __float_as_uint(__uint_as_float(r0[k]) * alpha);
                    r1[k] = __float_as_uint(__uint_as_float(r1[k]) * alpha);
                }
                ptx::tmem_st32(tmem + lb + TM_O + 32 * c4, r0);
                ptx::tmem_st32(tmem + lb + TM_O + 32 * (c4 + 1), r1);
            }
        }
        {
            uint32_t p0[32], p1[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                p0[k] = pk[k];
                p1[k] = pk[32 + k];
            }
            ptx::tmem_st32(tmem + lb + TM_P + st * 64, p0);
            ptx::tmem_st32(tmem + lb + TM_P + st * 64 + 32, p1);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(fbar(base, F_PFULL + st));
    }
    if (!ok) return;
    const int jl = n_t - 1;
    if (!fwait_warp(fbar(base, F_PVDONE + (jl & 1)), (jl >> 1) & 1, wc, lane)) return;
    ptx::tc_fence_after();
    const bool live = q0 + i < a.n_queries;
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(a.o + ((size_t)(q0 + i) * a.n_h + h) * DH);
#pragma unroll 1
    for (int c4 = 0; c4 < DH / 32; ++c4) {
        uint32_t r[32];
        ptx::tmem_ld32(tmem + lb + TM_O + 32 * c4, r);
        ptx::tmem_wait_ld_regs(r);
        if (live) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint4 v;
                v.x = ptx::pack_bf16(__uint_as_float(r[8 * k + 0]) * inv_l, __uint_as_float(r[8 * k + 1]) * inv_l);
                v.y = ptx::pack_bf16(__uint_as_float(r[8 * k + 2]) * inv_l, __uint_as_float(r[8 * k + 3]) * inv_l);
                v.z = ptx::pack_bf16(__uint_as_float(r[8 * k + 4]) * inv_l, __uint_as_float(r[8 * k + 5]) * inv_l);
                v.w = ptx::pack_bf16(__uint_as_float(r[8 * k + 6]) * inv_l, __uint_as_float(r[8 * k + 7]) * inv_l);
                dst[4 * c4 + k] = v;
            }
        }
    }
    if (live) a.lse[(size_t)(q0 + i) * a.n_h + h] = l > 0.f ? (m + __log2f(l)) * LN2 : -INFINITY;
}

// grid: ceil(T / 128) * n_h CTAs, head-major (the query tiles of one head are adjacent, longest
// first), so that one head's K and V (4 MB at T = 8192) are read from DRAM about once and then
// from L2 by its other query tiles; with heads interleaved instead, every query tile fetched them
// again (ncu: 15.3 GB of DRAM reads per launch against 1.2 GB of algorithmic bytes)
__global__ void __launch_bounds__(NTHREADS, 1)
    flash_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmr, const __grid_constant__ CUtensorMap tmv, const FlashArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = ptx::smem_u32(smem);
    if (base & 1023u) {
        if (threadIdx.x == 0) set_device_error(MLA_ERR_UNSUPPORTED);
        return;
    }
    launch_dependents();
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = (a.n_queries + BQ - 1) / BQ;
    const int h = (int)(blockIdx.x / n_qt), qt = n_qt - 1 - (int)(blockIdx.x % n_qt);
    const int q0 = qt * BQ;
    const int n_t = key_tiles(a, q0);
    if (threadIdx.x == 0) {
        ptx::mbar_init(fbar(base, F_QFULL), 1);
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(fbar(base, F_KVFULL + b), 1);
            ptx::mbar_init(fbar(base, F_KVEMPTY + b), 1);
            ptx::mbar_init(fbar(base, F_SFULL + b), 1);
            ptx::mbar_init(fbar(base, F_SFREE + b), 4);
            ptx::mbar_init(fbar(base, F_PFULL + b), 4);
            ptx::mbar_init(fbar(base, F_PVDONE + b), 1);
        }
        ptx::mbar_init(fbar(base, F_DONE), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmq);
        ptx::prefetch_tmap(&tmk);
        ptx::prefetch_tmap(&tmr);
        ptx::prefetch_tmap(&tmv);
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + OFF_MISC, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const FWait wc{a.wait_ns, abort_flag, false};
    if (n_t > 0) {
        if (warp == 0) {
            if (lane == 0) f_producer(a, &tmq, &tmk, &tmr, &tmv, base, h, q0, n_t, wc);
        } else if (warp == 1) {
            f_mma(base, tmem, n_t, wc, lane);
        } else {
            f_softmax(a, base, tmem, h, q0, n_t, warp, lane, wc);
        }
    }
    // wait for the preceding grid before leaving, so that this grid's completion implies its own
    if (threadIdx.x == 0) grid_dependency_wait();
    ptx::tc_fence_before();
    __syncthreads();
    if (*abort_flag) {  // copies issued before an abort get time to land
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) {
        }
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// 2-D bf16 map over [rows, inner] with row pitch `pitch` elements; box 64 columns x 128 rows,
// 128-byte swizzle; reads past the extents return zeros.
inline bool encode_map(CUtensorMap* tm, const void* p, uint64_t inner, uint64_t rows, uint64_t pitch) {
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
    cuuint64_t strides[1] = {pitch * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace of the un-absorbed prefill, in bytes, each part 256-byte aligned: the gathered rows
// [L, W], K and V [L, n_h d_h], the query [n_h, T, d_h + d_r] (bf16).
struct UnabsorbedWs {
    size_t rows, k, v, qu, total;
};
inline UnabsorbedWs unabsorbed_ws(int n_h, int d_h, int d_r, int width, long long L, long long T) {
    auto al = [](size_t b) { return (b + 255) & ~(size_t)255; };
    UnabsorbedWs w;
    w.rows = 0;
    w.k = w.rows + al((size_t)L * width * 2);
    w.v = w.k + al((size_t)L * n_h * d_h * 2);
    w.qu = w.v + al((size_t)L * n_h * d_h * 2);
    w.total = w.qu + al((size_t)T * n_h * (d_h + d_r) * 2);
    return w;
}

}  // namespace tcf
}  // namespace mla
