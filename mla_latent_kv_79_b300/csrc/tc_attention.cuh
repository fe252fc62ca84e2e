// tcgen05 split attention over the paged latent cache (sm_103a fast path).
//
// Shapes: n_h = 128 heads, d_c = 512, d_r = 64 (W = 576), page = 64 tokens, bf16 operands,
// fp32 softmax and accumulation.  This is the absorbed decode of the MLA glossary page (the
// up-projection folded into the query and the output) over the latent cache of the
// operator-notes page, section 3: all heads attend to the same cached row [c_kv | k_rope].
//
// One unit of the split schedule (sched.cuh) runs on a cluster of two CTAs with different
// jobs, because one SM's 512 TMEM columns cannot hold both the query (288 columns of bf16
// pairs) and the 128 x 512 fp32 output accumulator:
//
//   score CTA (rank 0)  TMEM: Q [0,288), S double buffer [288,416)
//     S = Q . page^T over all 576 columns, issued by two warps taking alternate pages (warp 1
//     the even pages into score buffer 0, warp 6 the odd ones into buffer 1), online softmax
//     (running max raised only when it grows by more than 2^8: O and l share the stale max, so
//     the result is exact), then P (bf16, 16 KB) plus (alpha, l) per head are stored with
//     st.async straight into one of the value CTA's four P buffers, completing bytes on its
//     mbarrier.
//   value CTA (rank 1)  TMEM: O [0,512)
//     rescales O rows when alpha != 1, then O += P . page[:, 0:512] with P as the
//     shared-memory A operand; drains O / l at the end of every segment.
//
// Each CTA streams the page through its own TMA ring: the score CTA all 576 columns in 3
// stages, so that it recycles a stage right after its QK instead of holding it until the
// value CTA's PV; the value CTA the 512 latent columns in 2 stages, read while the lines are
// still in L2, which leaves room for four P buffers.  The score-to-value traffic is
// one-directional and four P buffers deep, so the st.async transfer and the release of a
// buffer back to the score CTA (each about a microsecond between SMs) stay off the pace.
//
// The query of a segment travels through the score CTA's ring too: two items of nine 64-row x
// 64-column boxes (144 KB, exactly two stages), so that the query and the segment's first page
// are in flight together.  The softmax warps (idle at a segment start) move their rows into
// TMEM with tcgen05.st, so the tensor pipe is not held up by the copy.
//
// Roles (224 threads per CTA): warp 0 TMA, warp 1 TMEM allocation and MMA issue, warps 2-5
// (one TMEM lane quarter each, one head per thread) softmax in the score CTA, rescale and
// drain in the value CTA; warp 6 issues the odd pages' score MMAs in the score CTA and hands P
// buffers back to the score CTA as their PVs complete in the value CTA.  Every wait is bounded.
//
// The MMA issuers run as whole warps: every lane computes the (warp-uniform) descriptors and
// one elected lane issues.  Issuing from a single active lane cost sub-partition issue slots
// that the softmax warps need (measured on B300: 8 % of the B=16 x 4096 decode and 20 % of the
// ragged B=256 one).
//
// In the score CTA the two issuers skip each other's pages, so a page's full barrier is one of
// (stage, issuer) and a query item's one of its stage: a parity wait is only unambiguous for a
// waiter that sees every phase of its barrier in order.
#pragma once

#include <cudaTypedefs.h>

#include "sched.cuh"
#include "simt_attention.cuh"
#include "mx_format.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace tca {

constexpr int NH = 128, DC = 512, DR = 64, WID = 576, PAGE = 64;
constexpr int CHUNK = 64 * 128;                   // 64 rows x 64 bf16, 128-byte swizzled
constexpr int LAT_CHUNKS = 8;
constexpr int MAX_STAGES = 3;
constexpr int S_STAGE_BYTES = 9 * CHUNK;          // score CTA: whole page, 9 chunks (72 KB)
constexpr int Q_ITEMS = 2;                        // ring items per query, nine 8 KB boxes each
constexpr int V_STAGE_BYTES = LAT_CHUNKS * CHUNK; // value CTA: latent part (64 KB)
constexpr int P_BYTES = NH * 128;                 // P [128 heads x 64 tokens] bf16, SW128 K-major
constexpr int META_BYTES = NH * 8;                // (alpha, l) per head, fp32
constexpr int PBUF_BYTES = P_BYTES + META_BYTES;
constexpr int MAX_PBUF = 4;
constexpr int HALF = 32;                          // MX caches: cache rows per raw item (half a page)
constexpr int MAX_RAW = 6;
enum {
    B_FULL = 0,                      // [STAGES] item landed: a page (value CTA) or a query item (score CTA)
    B_EMPTY = B_FULL + MAX_STAGES,   // [STAGES] this CTA's consumer released the stage
    B_SFULL = B_EMPTY + MAX_STAGES,  // [2] score CTA: S buffer written
    B_SFREE = B_SFULL + 2,           // [2] score CTA: S buffer read by the 4 softmax warps
    B_PFULL = B_SFREE + 2,           // [NPBUF] value CTA: P + meta landed (own expect_tx + bytes)
    B_PEMPTY = B_PFULL + MAX_PBUF,   // [NPBUF] score CTA: value CTA's PV finished with P buffer b
    B_PREADY = B_PEMPTY + MAX_PBUF,  // [NPBUF] value CTA: O rescaled, P buffer b ready for the MMA
    B_PVDONE = B_PREADY + MAX_PBUF,  // [NPBUF] value CTA: PV of the page that used P buffer b complete
    B_OFREE = B_PVDONE + MAX_PBUF,   // value CTA: O drained
    B_DONE = B_OFREE + 1,            // MMA drain at exit
    B_QREADY = B_DONE + 1,           // score CTA: the segment's query is in TMEM (4 softmax warps)
    B_RFULL = B_QREADY + 1,          // MX caches: [RAW_STAGES] raw half page landed
    B_REMPTY = B_RFULL + MAX_RAW,    // MX caches: [RAW_STAGES] the 4 converter warps read it
    B_FULLP = B_REMPTY + MAX_RAW,    // score CTA: [STAGES][2] page of issuer i landed in a stage
    B_QSEEN = B_FULLP + 2 * MAX_STAGES,  // score CTA: both issuers saw the segment's query
    B_DRYW = B_QSEEN + 1,            // never arrived on: a parity-1 wait passes (the dry pass)
    B_DRYC = B_DRYW + 1,             // arrivals of the dry pass, never waited on
    NBARS = B_DRYC + 1
};
static_assert(NBARS <= 64, "the producer tracks full barriers in 64-bit masks");

// Shared-memory layout per cache format (KVF: KV_PLAIN, KV_MXFP8, KV_MXFP4).  Both CTAs of a
// pair use the same offsets.  The plain cache streams bf16 pages by TMA into a 3-stage ring in
// the score CTA and a 2-stage one (the latent columns) in the value CTA, which keeps four P
// buffers.  An MX cache streams raw half pages (codes, then the 32 rows' scale bytes) by bulk
// copy into a raw ring; four converter warps widen them into a 2-stage bf16 ring of the same
// layout as the TMA writes, so the MMA and softmax code is shared (two P buffers: the raw
// ring takes the rest of shared memory).
template <int KVF>
struct Lay {
    static constexpr int STAGES = KVF == KV_PLAIN ? 3 : 2;         // score CTA ring
    static constexpr int VSTAGES = 2;                              // value CTA ring
    static constexpr int NPBUF = KVF == KV_PLAIN ? 4 : 2;          // P buffers in the value CTA
    static constexpr int R_BYTES = NPBUF * PBUF_BYTES;
    static constexpr int OFF_R = VSTAGES * V_STAGE_BYTES;          // value CTA: P buffers
    static constexpr int ROW_BYTES = KVF == KV_MXFP4 ? WID / 2 : WID;  // code bytes per cache row
    static constexpr int RAW_CODES = HALF * ROW_BYTES;
    static constexpr int RAW_SCALES = HALF * (WID / MX_BLOCK);
    static constexpr int RAW_STAGE = (RAW_CODES + RAW_SCALES + 127) & ~127;
    static constexpr int RAW_STAGES = KVF == KV_MXFP4 ? 6 : (KVF == KV_MXFP8 ? 3 : 0);
    static constexpr int RAW_RING = RAW_STAGES > 0 ? RAW_STAGES : 1;  // ring arithmetic (MX only)
    static constexpr int RING_END = STAGES * S_STAGE_BYTES > OFF_R + R_BYTES ? STAGES * S_STAGE_BYTES
                                                                             : OFF_R + R_BYTES;
    static constexpr int OFF_RAW = RING_END;
    static constexpr int OFF_BARS = OFF_RAW + RAW_STAGES * RAW_STAGE;
    static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;
    static constexpr int OFF_RED = OFF_MISC + 16;                  // schedule scratch
    static constexpr int SMEM_BYTES = OFF_RED + SCHED_SCRATCH * 8;
    static constexpr int NTHREADS = KVF == KV_PLAIN ? 224 : 352;   // + 4 converter warps
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(RAW_STAGES <= MAX_RAW, "raw ring barriers");
    static_assert(NPBUF <= MAX_PBUF && VSTAGES <= MAX_STAGES, "ring barriers");
    static_assert(KVF == KV_PLAIN || VSTAGES == STAGES, "the MX converters run one ring depth in both CTAs");
    static_assert(RAW_CODES % 16 == 0 && RAW_SCALES % 16 == 0, "bulk copies move multiples of 16 bytes");
};
constexpr int TM_Q = 0, TM_S = 288, TM_O = 0;
constexpr float TAU = 8.0f;  // log2 units
constexpr float LN2 = 0.6931471805599453f;
constexpr uint32_t IDESC_QK = ptx::idesc_bf16(128, 64, false, false);
constexpr uint32_t IDESC_PV = ptx::idesc_bf16(128, 256, false, true);

struct TcArgs {
    AttnArgs a;
    unsigned long long wait_ns;
    float scale_log2;
};

struct WaitCtl {
    unsigned long long limit_ns;
    volatile int* abort;
    bool ignore_abort;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl& w, bool cluster_scope = false) {
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
        if (i & 1u) {  // every second failed poll (try_wait itself may suspend the thread)
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

// Warp-uniform bounded wait: every lane observes the phase (acquire), all lanes leave together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w, bool cluster_scope,
                                          int lane) {
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const bool ok = cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if (i & 1u) {  // every second failed poll (try_wait itself may suspend the thread)
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

template <int KVF>
__device__ __forceinline__ uint32_t bar_addr(uint32_t base, int i) {
    return base + Lay<KVF>::OFF_BARS + 8u * (uint32_t)i;
}

// The full barrier of a ring item and the bit that tracks its parity in a waiter's or filler's
// 32-bit mask: a query item's is its stage's (score CTA) and a page's is (stage, page parity)
// in the score CTA, its stage's in the value CTA.
__device__ __forceinline__ int full_index(uint32_t rank, bool query, uint32_t stage, uint32_t page) {
    return (rank == 0 && !query) ? B_FULLP + 2 * (int)stage + (int)(page & 1u) : B_FULL + (int)stage;
}

// ----------------------------------------------------------------------------- warp 0: TMA
// Both CTAs run the same page sequence.  Plain cache: the score CTA loads the segment's query
// and then all nine 64-column chunks of each page, the value CTA the eight latent chunks, by
// tensor TMA into the bf16 ring.  MX cache: both CTAs bulk-copy each page as two raw half pages
// (32 rows of codes, then their scale bytes, both contiguous in the pool) into the raw ring; the
// converter warps fill every item of the bf16 ring, the query's too (a parity wait on a ring
// barrier is only unambiguous for a party that fills every item of the ring in order).
template <int KVF, int STAGES>  // STAGES: depth of this CTA's bf16 ring
__device__ __forceinline__ void producer(const AttnArgs& a, const CUtensorMap* tm, const CUtensorMap* tmq, UnitCursor c,
                                         uint32_t base, uint32_t rank, const WaitCtl& wc) {
    using L = Lay<KVF>;
    uint32_t g = 0;       // plain cache: bf16 ring items (queries and pages), in ring order
    uint32_t gp = 0;      // pages
    uint32_t r = 0;       // MX cache: raw items issued
    uint64_t fpar = 0;    // plain cache: parity of the next phase of each full barrier (bit = index)
    uint64_t armed = 0;   // plain cache: full barriers armed at least once
    bool ok = true;
    Segment sg;
    const int nch = rank == 0 ? 9 : LAT_CHUNKS;
    const uint32_t stage_bytes = (uint32_t)(nch * CHUNK);
    bool waited = false;
    while (ok && c.next(a.qs, &sg)) {
        const int pg0 = sg.page_begin;
        if (!waited) {
            // The kernels before this one in the stream may still be running (programmatic
            // launch): the absorption GEMM writes the queries, and an earlier cache append may
            // not have finished either, so the first load waits for the preceding grid.
            // (Issuing the unit's first page, or an L2 prefetch of it, before this wait
            // measured no faster.)
            grid_dependency_wait();
            waited = true;
        }
        if (KVF == KV_PLAIN && rank == 0) {  // the segment's query: box b of the 18 is (columns 64*(b/2), rows 64*(b%2))
            for (int qi = 0; qi < Q_ITEMS; ++qi, ++g) {
                const uint32_t stage = g % STAGES;
                if (!wait_bar(bar_addr<KVF>(base, B_EMPTY + stage), ((g / STAGES) & 1u) ^ 1u, wc)) { ok = false; break; }
                const int fi = full_index(rank, true, stage, gp);
                const uint32_t fb = bar_addr<KVF>(base, fi), dst = base + stage * S_STAGE_BYTES;
                fpar ^= 1ull << fi;
                armed |= 1ull << fi;
                ptx::mbar_arrive_expect_tx(fb, (uint32_t)S_STAGE_BYTES);
                for (int j = 0; j < 9; ++j) {
                    const int b = 9 * qi + j;
                    ptx::tma_load_2d(dst + j * CHUNK, tmq, (b >> 1) * 64, sg.q * NH + (b & 1) * 64, fb);
                }
            }
            if (!ok) break;
        }
        for (int pg = pg0; pg < sg.page_end; ++pg, ++g, ++gp) {
            int page = __ldg(a.page_table + (long long)sg.seq * a.max_pages + pg);
            if (page < 0 || page >= a.num_pages) {
                set_device_error(MLA_ERR_DEVICE_BOUNDS);
                page = 0;  // keep the pipeline fed; the result of this query is void
            }
            if (KVF == KV_PLAIN) {
                const uint32_t stage = g % STAGES;
                if (!wait_bar(bar_addr<KVF>(base, B_EMPTY + stage), ((g / STAGES) & 1u) ^ 1u, wc)) { ok = false; break; }
                const int fi = full_index(rank, false, stage, gp);
                const uint32_t fb = bar_addr<KVF>(base, fi);
                fpar ^= 1ull << fi;
                armed |= 1ull << fi;
                ptx::mbar_arrive_expect_tx(fb, stage_bytes);
                const uint32_t dst = base + stage * stage_bytes;
                for (int cc = 0; cc < nch; ++cc) ptx::tma_load_2d(dst + cc * CHUNK, tm, cc * 64, page * PAGE, fb);
            } else {
                for (int hf = 0; hf < 2; ++hf, ++r) {
                    const uint32_t rs = r % L::RAW_RING;
                    if (!wait_bar(bar_addr<KVF>(base, B_REMPTY + rs), ((r / L::RAW_RING) & 1u) ^ 1u, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_addr<KVF>(base, B_RFULL + rs);
                    const uint32_t dst = base + L::OFF_RAW + rs * L::RAW_STAGE;
                    const long long row0 = (long long)page * PAGE + hf * HALF;
                    ptx::mbar_arrive_expect_tx(fb, (uint32_t)(L::RAW_CODES + L::RAW_SCALES));
                    ptx::bulk_load(dst, reinterpret_cast<const uint8_t*>(a.pool) + row0 * L::ROW_BYTES,
                                   (uint32_t)L::RAW_CODES, fb);
                    ptx::bulk_load(dst + L::RAW_CODES, reinterpret_cast<const uint8_t*>(a.scales) + row0 * (WID / MX_BLOCK),
                                   (uint32_t)L::RAW_SCALES, fb);
                }
                if (!ok) break;
            }
        }
    }
    if (!ok) {  // let loads already in flight land before the CTA leaves
        WaitCtl w2 = wc;
        w2.ignore_abort = true;
        w2.limit_ns = 20000000ull;
        if (KVF == KV_PLAIN) {  // the last phase armed on each full barrier
            for (int i = 0; i < NBARS; ++i)
                if ((armed >> i) & 1ull) wait_bar(bar_addr<KVF>(base, i), (uint32_t)((fpar >> i) & 1ull) ^ 1u, w2);
        } else {
            for (uint32_t k = r > (uint32_t)L::RAW_RING ? r - L::RAW_RING : 0u; k < r; ++k)
                wait_bar(bar_addr<KVF>(base, B_RFULL + k % L::RAW_RING), (k / L::RAW_RING) & 1u, w2);
        }
    }
}

// ----------------------------------------------------------------------------- MX converters
// Warps 7-10 of both CTAs (MX caches only) fill every item of the bf16 ring, in order, each
// warp waiting for the item's stage to be free and arriving on its full barrier (count 4).
// Score CTA, the segment's query: warp 7 loads its two items by tensor TMA (the same 18 boxes
// as a plain cache), completing their bytes on the full barrier.  Every page: the warps widen
// its two raw half pages into the stage.  Item = (row, 16-byte group of
// codes): an MXFP8 group is 16 codes of half a block, an MXFP4 group 32 codes of one block.
// Each code becomes code value * 2^(scale byte - 127) in bf16, exactly, written at the place the
// 128-byte-swizzled TMA layout gives it (64-column chunk, row, 16-byte piece p at
// (p ^ (row & 7)) * 16).  Rows past the sequence end are written as zeros, so that whatever
// bytes the pool holds there meet a zero weight as zeros.  The score CTA converts all 576
// columns, the value CTA the 512 latent ones.
template <int KVF>
__device__ __forceinline__ void converter(const AttnArgs& a, const CUtensorMap* tmq, UnitCursor c, uint32_t base,
                                          uint32_t rank, int cw, int lane, const WaitCtl& wc) {
    using L = Lay<KVF>;
    constexpr int STAGES = L::STAGES;
    constexpr int GC = KVF == KV_MXFP4 ? 32 : 16;   // codes per 16-byte group
    constexpr int NW = GC / 2;                      // bf16 pairs per group
    constexpr int SB = WID / MX_BLOCK;              // scale bytes per row
    const int G = (rank == 0 ? WID : DC) / GC;      // groups of a row this CTA converts
    const int n_items = HALF * G;
    const int ctid = cw * 32 + lane;
    const uint32_t stage_bytes = rank == 0 ? S_STAGE_BYTES : V_STAGE_BYTES;
    uint32_t k = 0, r = 0, gp = 0;  // bf16 ring items, raw items, pages
    uint32_t qpar = 0, qarmed = 0;  // warp 7: next phase parity / armed, per stage, of the query barriers
    bool ok = true, waited = false;
    Segment sg;
    while (ok && c.next(a.qs, &sg)) {
        if (rank == 0) {
            if (cw == 0 && lane == 0 && !waited) {
                grid_dependency_wait();  // the query comes from the kernel before this one
                waited = true;
            }
            for (int qi = 0; qi < Q_ITEMS; ++qi, ++k) {
                const uint32_t stage = k % STAGES;
                if (!warp_wait(bar_addr<KVF>(base, B_EMPTY + stage), ((k / STAGES) & 1u) ^ 1u, wc, false, lane)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = bar_addr<KVF>(base, B_FULL + stage);
                if (lane == 0) {
                    if (cw == 0) {  // box b of the 18 is (columns 64*(b/2), rows 64*(b%2))
                        const uint32_t dst = base + stage * S_STAGE_BYTES;
                        ptx::mbar_arrive_expect_tx(fb, (uint32_t)S_STAGE_BYTES);
                        for (int j = 0; j < 9; ++j) {
                            const int b = 9 * qi + j;
                            ptx::tma_load_2d(dst + j * CHUNK, tmq, (b >> 1) * 64, sg.q * NH + (b & 1) * 64, fb);
                        }
                        qpar ^= 1u << stage;
                        qarmed |= 1u << stage;
                    } else {
                        ptx::mbar_arrive(fb);
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        for (int pg = sg.page_begin; pg < sg.page_end; ++pg, ++k, ++gp) {
            const uint32_t stage = k % STAGES;
            if (!warp_wait(bar_addr<KVF>(base, B_EMPTY + stage), ((k / STAGES) & 1u) ^ 1u, wc, false, lane)) {
                ok = false;
                break;
            }
            const uint32_t dst = base + stage * stage_bytes;
            const int valid = sg.len - pg * PAGE;  // rows of this page that hold tokens
            for (int hf = 0; hf < 2; ++hf, ++r) {
                const uint32_t rs = r % L::RAW_RING;
                if (!warp_wait(bar_addr<KVF>(base, B_RFULL + rs), (r / L::RAW_RING) & 1u, wc, false, lane)) {
                    ok = false;
                    break;
                }
                const uint32_t raw = base + L::OFF_RAW + rs * L::RAW_STAGE;
#pragma unroll 1
                for (int i = ctid; i < n_items; i += 128) {
                    const int row = i / G, grp = i - row * G;
                    const int trow = hf * HALF + row;
                    const uint4 cv = ptx::ld_shared_v4u(raw + (uint32_t)(row * L::ROW_BYTES + grp * 16));
                    const int blk = KVF == KV_MXFP4 ? grp : (grp >> 1);
                    const float sc = exp2_int((int)ptx::ld_shared_u8(raw + (uint32_t)(L::RAW_CODES + row * SB + blk)) - 127);
                    const uint32_t cw4[4] = {cv.x, cv.y, cv.z, cv.w};
                    uint32_t w[NW];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (KVF == KV_MXFP8) {
                            const float2 lo = e4m3x2_to_f32(cw4[j] & 0xFFFFu), hi = e4m3x2_to_f32(cw4[j] >> 16);
                            w[2 * j] = ptx::pack_bf16(lo.x * sc, lo.y * sc);
                            w[2 * j + 1] = ptx::pack_bf16(hi.x * sc, hi.y * sc);
                        } else {
#pragma unroll
                            for (int bb = 0; bb < 4; ++bb) {
                                const float2 v = e2m1x2_to_f32(cw4[j] >> (8 * bb));
                                w[4 * j + bb] = ptx::pack_bf16(v.x * sc, v.y * sc);
                            }
                        }
                    }
                    if (trow >= valid) {
#pragma unroll
                        for (int q = 0; q < NW; ++q) w[q] = 0u;
                    }
                    // GC codes = GC bf16 = GC / 8 pieces of 16 bytes, starting at column grp * GC
                    const int cc = (grp * GC) >> 6, p0 = ((grp * GC) & 63) >> 3;
                    const uint32_t rowp = dst + (uint32_t)(cc * CHUNK + trow * 128);
#pragma unroll
                    for (int q = 0; q < GC / 8; ++q)
                        ptx::st_shared_v4(rowp + ((uint32_t)((p0 + q) ^ (trow & 7)) << 4), w[4 * q], w[4 * q + 1],
                                          w[4 * q + 2], w[4 * q + 3]);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, B_REMPTY + rs));
            }
            if (!ok) break;
            ptx::fence_proxy_async();  // the tensor core reads the stage through the async proxy
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, full_index(rank, false, stage, gp)));
        }
    }
    if (!ok && cw == 0 && lane == 0) {  // let query loads still in flight land (bounded)
        WaitCtl w2 = wc;
        w2.ignore_abort = true;
        w2.limit_ns = 20000000ull;
        for (int st = 0; st < STAGES; ++st)
            if ((qarmed >> st) & 1u) wait_bar(bar_addr<KVF>(base, B_FULL + st), ((qpar >> st) & 1u) ^ 1u, w2);
    }
}

// ----------------------------------------------------------------------------- score CTA
// Two issuing warps (warps 1 and 6, one elected lane issuing) split the pages: ISSUER takes the
// pages with page index % 2 == ISSUER, always into score buffer ISSUER.  One thread issuing all
// 36 MMAs of a page was the pace setter (about 88 cycles per N=64 MMA beside the softmax
// warps).  Each waits only on its own barriers: a page's full barrier of (stage, issuer), its
// score buffer's free barrier, and the query barriers, which both see every phase of (QSEEN
// keeps the next query out of TMEM until both saw this one).
template <int KVF, int ISSUER>
__device__ __forceinline__ void score_mma(const AttnArgs& a, UnitCursor c, uint32_t base, uint32_t tmem,
                                          const WaitCtl& wc, int lane) {
    constexpr int STAGES = Lay<KVF>::STAGES;
    constexpr uint32_t sb = ISSUER;
    const uint32_t dry_w = bar_addr<KVF>(base, B_DRYW), dry_c = bar_addr<KVF>(base, B_DRYC);
    uint32_t g = 0, k = 0, segn = 0;  // pages, ring items, segments
    uint32_t pbits = 0;               // parity of the next phase of this issuer's page barrier, per stage
    uint32_t uses = 0;                // pages issued into this issuer's score buffer
    int pg = 0, pend = 0;             // the open segment's pages
    bool ok = true;
    // The first pass is dry: the page body runs once at entry, on whatever the score buffer,
    // the query columns and stage 0 hold, against barriers that pass at once or that nobody
    // waits on.  Its code is then in the instruction caches when the first page lands (after
    // an L2 flush that first pass costs several microseconds); the first real MMA of the
    // buffer overwrites what it wrote, and the drain commit below covers its MMAs.
    bool dry = true;
    Segment sg;
    for (;;) {
        uint32_t stage = 0;
        if (!dry) {
            // this issuer's next page, opening segments as the cursor yields them
            bool found = false;
            while (!found) {
                if (pg >= pend) {
                    if (!c.next(a.qs, &sg)) break;
                    // the softmax warps put the segment's query into TMEM columns [TM_Q,
                    // TM_Q + 288) (they do so only after reading the previous segment's last
                    // scores, i.e. after its QKs); then the stages that carried it are free
                    if (!warp_wait(bar_addr<KVF>(base, B_QREADY), segn & 1u, wc, false, lane)) { ok = false; break; }
                    ptx::tc_fence_after();
                    if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, B_QSEEN));
                    if (ISSUER == 0)
                        for (int qi = 0; qi < Q_ITEMS; ++qi)
                            if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, B_EMPTY + (k + qi) % STAGES));
                    k += Q_ITEMS;
                    ++segn;
                    pg = sg.page_begin;
                    pend = sg.page_end;
                    continue;
                }
                if ((g & 1u) == sb) found = true;
                else ++pg, ++g, ++k;  // the other issuer's page
            }
            if (!ok || !found) break;
            stage = k % STAGES;
        }
        const uint32_t bfull = dry ? dry_w : bar_addr<KVF>(base, B_FULLP + 2 * stage + sb);
        if (!warp_wait(bfull, dry ? 1u : (pbits >> stage) & 1u, wc, false, lane)) break;
        const uint32_t bsfree = dry ? dry_w : bar_addr<KVF>(base, B_SFREE + sb);
        if (!warp_wait(bsfree, dry ? 1u : (uses & 1u) ^ 1u, wc, false, lane)) break;
        pbits ^= dry ? 0u : 1u << stage;
        uses += dry ? 0u : 1u;
        ptx::tc_fence_after();
        // descriptors are the stage's base descriptor plus compile-time offsets (the 14-bit
        // address field cannot carry: shared addresses are < 256 KB).  The 36 MMAs are fully
        // unrolled: with a loop around them the issuing thread, not the tensor core, set the
        // pace (measured on B300 with one issuing lane: about 85 cycles per N=64 MMA against
        // 48 unrolled).
        const uint64_t d_pg = ptx::desc_sw128(base + stage * S_STAGE_BYTES, 16, 1024);
        const uint32_t d = tmem + TM_S + sb * 64;
#pragma unroll
        for (int cc = 0; cc < 9; ++cc) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA, 4 per 64-column chunk
                ptx::mma_ts_elect(d, tmem + TM_Q + cc * 32 + kk * 8, d_pg + (uint64_t)((cc * CHUNK + kk * 32) >> 4),
                                  IDESC_QK, (cc | kk) ? 1u : 0u);
        }
        ptx::tc_commit_elect(dry ? dry_c : bar_addr<KVF>(base, B_SFULL + sb));
        ptx::tc_commit_elect(dry ? dry_c : bar_addr<KVF>(base, B_EMPTY + stage));
        if (!dry) ++pg, ++g, ++k;
        dry = false;
    }
    // every MMA this thread issued completes before the CTA frees its TMEM (the drain barrier
    // counts both issuers): a fixed 20 ms bound, whatever the configured limit (which may be
    // microseconds when a caller tests timeouts)
    __syncwarp();
    ptx::tc_commit_elect(bar_addr<KVF>(base, B_DONE));
    WaitCtl w2 = wc;
    w2.ignore_abort = true;
    w2.limit_ns = 20000000ull;
    warp_wait(bar_addr<KVF>(base, B_DONE), 0, w2, false, lane);
}

template <int KVF>
__device__ __forceinline__ void score_softmax(const TcArgs& args, UnitCursor c, uint32_t base, uint32_t tmem,
                                              uint32_t peer, int warp, int lane, const WaitCtl& wc) {
    constexpr int STAGES = Lay<KVF>::STAGES;
    constexpr int OFF_R = Lay<KVF>::OFF_R;
    constexpr uint32_t NPBUF = Lay<KVF>::NPBUF;
    const AttnArgs& a = args.a;
    const int qd = warp & 3;  // TMEM lane quarter this warp may access
    const int h = qd * 32 + lane;
    const uint32_t lb = (uint32_t)(qd * 32) << 16;
    const uint32_t tS = tmem + lb + TM_S, tQ = tmem + lb + TM_Q;
    const uint32_t pbuf_r = ptx::mapa(base + OFF_R, peer);          // value CTA's P buffers
    const uint32_t pfull_r = ptx::mapa(bar_addr<KVF>(base, B_PFULL), peer);
    const uint32_t sw = (uint32_t)(h & 7);
    uint32_t g = 0, k = 0, segn = 0;  // pages, ring items, segments
    uint32_t qbits = 0;               // parity of the next phase of each stage's query barrier
    bool ok = true;
    Segment sg;
    while (ok && c.next(a.qs, &sg)) {
        // this thread's query row (head h) from the two ring items into TMEM: 64-column chunk c
        // of the row is 128 swizzled bytes (16-byte piece p at (p ^ (h & 7)) * 16) of box
        // 2c + h/64, i.e. 32 columns of bf16 pairs
        for (int qi = 0; qi < Q_ITEMS && ok; ++qi, ++k) {
            const uint32_t stage = k % STAGES;
            if (!warp_wait(bar_addr<KVF>(base, B_FULL + stage), (qbits >> stage) & 1u, wc, false, lane)) { ok = false; break; }
            qbits ^= 1u << stage;
#pragma unroll 1
            for (int j = 0; j < 9; ++j) {
                const int b = 9 * qi + j;
                if ((b & 1) != (h >> 6)) continue;  // warp-uniform: a quarter's heads share h / 64
                const uint32_t row = base + stage * S_STAGE_BYTES + j * CHUNK + (uint32_t)(h & 63) * 128u;
                uint32_t r[32];
#pragma unroll
                for (int pc = 0; pc < 8; ++pc) {
                    const float4 v = ptx::ld_shared_v4(row + ((pc ^ sw) << 4));
                    r[4 * pc + 0] = __float_as_uint(v.x);
                    r[4 * pc + 1] = __float_as_uint(v.y);
                    r[4 * pc + 2] = __float_as_uint(v.z);
                    r[4 * pc + 3] = __float_as_uint(v.w);
                }
                ptx::tmem_st32(tQ + (b >> 1) * 32, r);
            }
        }
        if (!ok) break;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        // both issuers saw the previous query's barrier phase, so none of them can find this
        // one two phases ahead
        if (segn > 0 && !warp_wait(bar_addr<KVF>(base, B_QSEEN), (segn - 1) & 1u, wc, false, lane)) { ok = false; break; }
        ++segn;
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, B_QREADY));
        float m_run = -INFINITY, l = 0.f;
        for (int pg = sg.page_begin; pg < sg.page_end; ++pg, ++g, ++k) {
            const uint32_t sb = g & 1u, use = g >> 1;
            if (!warp_wait(bar_addr<KVF>(base, B_SFULL + sb), use & 1u, wc, false, lane)) { ok = false; break; }
            ptx::tc_fence_after();
            float s[64];
            {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(tS + sb * 64, r0);
                ptx::tmem_ld32(tS + sb * 64 + 32, r1);
                ptx::tmem_wait_ld_regs(r0);
                ptx::tmem_wait_ld_regs(r1);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = __uint_as_float(r0[j]);
                    s[32 + j] = __uint_as_float(r1[j]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, B_SFREE + sb));

            // raw scores; tokens past the sequence end are masked (only the last page of a
            // sequence has any, and the branch is warp-uniform).  The scale (log2 units) is
            // positive, so it scales the maximum and folds into the exponent's FFMA.
            const int valid = sg.len - pg * PAGE;
            if (valid < PAGE) {
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (j >= valid) s[j] = -INFINITY;
            }
            float mr = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) mr = fmaxf(mr, s[j]);
            const float c2 = args.scale_log2;
            const float mx = mr * c2;
            float alpha = 1.f;
            if (mx > m_run + TAU) {
                alpha = ptx::ex2(m_run - mx);
                m_run = mx;
                l *= alpha;
            }
            float sum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = ptx::ex2(fmaf(s[2 * j], c2, -m_run)), p1 = ptx::ex2(fmaf(s[2 * j + 1], c2, -m_run));
                sum += p0 + p1;
                pk[j] = ptx::pack_bf16(p0, p1);
            }
            l += sum;
            // P row h -> value CTA, 128-byte swizzled (16-byte chunk k at k ^ (h & 7)).  P
            // buffers come back in page order (the PVs complete in order and one warp hands them
            // back), so an even page waits for the next page's buffer, which covers its own, and
            // an odd page waits for nothing: one wait per two pages, always on the odd buffers,
            // each of which sees every phase.
            const uint32_t pb = g % NPBUF;
            if ((g & 1u) == 0) {
                const uint32_t gn = g + 1;
                if (!warp_wait(bar_addr<KVF>(base, B_PEMPTY + gn % NPBUF), ((gn / NPBUF) & 1u) ^ 1u, wc, true, lane)) {
                    ok = false;
                    break;
                }
            }
            const uint32_t row = pbuf_r + pb * PBUF_BYTES + (uint32_t)h * 128u;
            const uint32_t fb = pfull_r + 8u * pb;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                ptx::st_async_v4_b32(row + ((c ^ sw) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3], fb);
            ptx::st_async_v2_f32(pbuf_r + pb * PBUF_BYTES + P_BYTES + (uint32_t)h * 8u, alpha, l, fb);
        }
        if (!ok) break;
        const float lse = l > 0.f ? (m_run + __log2f(l)) * LN2 : -INFINITY;
        if (sg.direct) a.lse[(size_t)sg.q * NH + h] = lse;
        else a.part_lse[(size_t)sg.slot * NH + h] = lse;
    }
}

// ----------------------------------------------------------------------------- value CTA
template <int KVF>
__device__ __forceinline__ void value_mma(const AttnArgs& a, UnitCursor c, uint32_t base, uint32_t tmem,
                                          const WaitCtl& wc, int lane) {
    constexpr int STAGES = Lay<KVF>::VSTAGES;
    constexpr int OFF_R = Lay<KVF>::OFF_R;
    constexpr uint32_t NPBUF = Lay<KVF>::NPBUF;
    const uint32_t dry_w = bar_addr<KVF>(base, B_DRYW), dry_c = bar_addr<KVF>(base, B_DRYC);
    uint32_t g = 0, segn = 0;  // pages, segments opened
    int pg = 0, pbeg = 0, pend = 0;
    // The first pass is dry (as in the score issuers): one page's PV on whatever P buffer 0 and
    // stage 0 hold, into O, which the first real page overwrites (its first MMA does not
    // accumulate); the drain commit below covers it.
    bool dry = true;
    Segment sg;
    for (;;) {
        if (!dry) {
            bool more = true;
            while (pg >= pend) {
                if (!c.next(a.qs, &sg)) { more = false; break; }
                pg = pbeg = sg.page_begin;
                pend = sg.page_end;
                ++segn;
            }
            if (!more) break;
        }
        const bool first = dry || pg == pbeg;
        const uint32_t stage = g % STAGES, pb = g % NPBUF;
        if (!warp_wait(dry ? dry_w : bar_addr<KVF>(base, B_FULL + stage), dry ? 1u : (g / STAGES) & 1u, wc, false, lane)) break;
        if (!warp_wait(dry ? dry_w : bar_addr<KVF>(base, B_PREADY + pb), dry ? 1u : (g / NPBUF) & 1u, wc, false, lane)) break;
        // O of the previous segment is drained before this segment's first PV overwrites it
        if (!dry && first && segn > 1 && !warp_wait(bar_addr<KVF>(base, B_OFREE), (segn - 2) & 1u, wc, false, lane)) break;
        ptx::tc_fence_after();
        const uint64_t da = ptx::desc_sw128(base + OFF_R + pb * PBUF_BYTES, 16, 1024);
        const uint64_t db = ptx::desc_sw128(base + stage * V_STAGE_BYTES, CHUNK, 1024);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // 16 tokens per MMA; V is MN-major: chunks 8 KB apart
                ptx::mma_ss_elect(tmem + TM_O + hf * 256, da + (uint64_t)((kk * 32) >> 4),
                                  db + (uint64_t)((hf * 4 * CHUNK + kk * 2048) >> 4), IDESC_PV,
                                  (first && kk == 0) ? 0u : 1u);
        }
        ptx::tc_commit_elect(dry ? dry_c : bar_addr<KVF>(base, B_PVDONE + pb));
        ptx::tc_commit_elect(dry ? dry_c : bar_addr<KVF>(base, B_EMPTY + stage));
        if (!dry) ++pg, ++g;
        dry = false;
    }
    // every MMA this thread issued completes before the CTA frees its TMEM: a fixed 20 ms bound,
    // whatever the configured limit (which may be microseconds when a caller tests timeouts)
    __syncwarp();
    ptx::tc_commit_elect(bar_addr<KVF>(base, B_DONE));
    WaitCtl w2 = wc;
    w2.ignore_abort = true;
    w2.limit_ns = 20000000ull;
    warp_wait(bar_addr<KVF>(base, B_DONE), 0, w2, false, lane);
}

template <int KVF>
__device__ __forceinline__ void value_warps(const AttnArgs& a, UnitCursor c, uint32_t base, uint32_t tmem, int warp,
                                            int lane, const WaitCtl& wc) {
    constexpr int OFF_R = Lay<KVF>::OFF_R;
    constexpr uint32_t NPBUF = Lay<KVF>::NPBUF;
    const int qd = warp & 3;
    const int h = qd * 32 + lane;
    const uint32_t tO = tmem + ((uint32_t)(qd * 32) << 16) + TM_O;
    uint32_t g = 0;
    bool ok = true;
    Segment sg;
    while (ok && c.next(a.qs, &sg)) {
        float l_last = 0.f;
        for (int pg = sg.page_begin; pg < sg.page_end; ++pg, ++g) {
            const bool first = pg == sg.page_begin;
            const uint32_t pb = g % NPBUF, use = g / NPBUF;
            if (warp == 2 && lane == 0) ptx::mbar_arrive_expect_tx(bar_addr<KVF>(base, B_PFULL + pb), PBUF_BYTES);
            if (!warp_wait(bar_addr<KVF>(base, B_PFULL + pb), use & 1u, wc, true, lane)) { ok = false; break; }
            const float2 meta = ptx::ld_shared_v2(base + OFF_R + pb * PBUF_BYTES + P_BYTES + (uint32_t)h * 8u);
            l_last = meta.y;
            const bool resc = !first && meta.x != 1.f;
            if (__any_sync(0xffffffffu, resc)) {
                // O must be stable: the previous page's PV has completed.  pvdone is kept per P
                // buffer so that no parity wait here is ever two phases away from its target
                // (P of this page was sent after the PV of page g - NPBUF completed).
                const uint32_t gp = g - 1;
                if (!warp_wait(bar_addr<KVF>(base, B_PVDONE + gp % NPBUF), (gp / NPBUF) & 1u, wc, false, lane)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const float alpha = resc ? meta.x : 1.f;
#pragma unroll 1
                for (int k0 = 0; k0 < 16; k0 += 2) {  // two loads in flight per wait
                    uint32_t r0[32], r1[32];
                    ptx::tmem_ld32(tO + 32 * k0, r0);
                    ptx::tmem_ld32(tO + 32 * (k0 + 1), r1);
                    ptx::tmem_wait_ld_regs(r0);
                    ptx::tmem_wait_ld_regs(r1);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        r0[j] = __float_as_uint(__uint_as_float(r0[j]) * alpha);
                        r1[j] = __float_as_uint(__uint_as_float(r1[j]) * alpha);
                    }
                    ptx::tmem_st32(tO + 32 * k0, r0);
                    ptx::tmem_st32(tO + 32 * (k0 + 1), r1);
                }
                ptx::tmem_wait_st();
            }
            ptx::fence_proxy_async();  // P arrived through the generic proxy; the MMA reads it via the async proxy
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, B_PREADY + pb));
        }
        if (!ok) break;
        // drain O / l once the segment's last PV has completed
        {
            const uint32_t gl = g - 1;
            if (!warp_wait(bar_addr<KVF>(base, B_PVDONE + gl % NPBUF), (gl / NPBUF) & 1u, wc, false, lane)) { ok = false; break; }
        }
        ptx::tc_fence_after();
        const float inv_l = l_last > 0.f ? 1.f / l_last : 0.f;
        // bf16 rows of O / l: the final output row o_lat[q][h][:], or the partial layout
        // [slot][c/8][h][8] in which a warp's 32 heads write 512 contiguous bytes.  Four TMEM
        // loads (128 columns) are in flight per wait: the load latency, not the stores, set the
        // pace when each 32-column load was waited for on its own.
        uint4* dst;
        size_t step;
        if (sg.direct) {
            dst = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(a.o_lat) + ((size_t)sg.q * NH + h) * DC);
            step = 1;
        } else {
            dst = reinterpret_cast<uint4*>(a.part_o) + (size_t)sg.slot * (DC / 8) * NH + h;
            step = NH;
        }
        auto emit = [&](const uint32_t* r, int k) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 v;
                v.x = ptx::pack_bf16(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l);
                v.y = ptx::pack_bf16(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l);
                v.z = ptx::pack_bf16(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l);
                v.w = ptx::pack_bf16(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l);
                dst[(size_t)(4 * k + i) * step] = v;
            }
        };
#pragma unroll 1
        for (int k0 = 0; k0 < 16; k0 += 4) {
            uint32_t r0[32], r1[32], r2[32], r3[32];
            ptx::tmem_ld32(tO + 32 * k0, r0);
            ptx::tmem_ld32(tO + 32 * (k0 + 1), r1);
            ptx::tmem_ld32(tO + 32 * (k0 + 2), r2);
            ptx::tmem_ld32(tO + 32 * (k0 + 3), r3);
            ptx::tmem_wait_ld_regs(r0);
            ptx::tmem_wait_ld_regs(r1);
            ptx::tmem_wait_ld_regs(r2);
            ptx::tmem_wait_ld_regs(r3);
            emit(r0, k0);
            emit(r1, k0 + 1);
            emit(r2, k0 + 2);
            emit(r3, k0 + 3);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_addr<KVF>(base, B_OFREE));
    }
}

// Value CTA, warp 6: as soon as the PV of page g has completed (its P buffer is read), tell the
// score CTA that the buffer may be refilled.  A warp of its own, so that the signal waits for
// nothing but that PV.
template <int KVF>
__device__ __forceinline__ void value_release(const AttnArgs& a, UnitCursor c, uint32_t base, int lane,
                                              const WaitCtl& wc) {
    constexpr uint32_t NPBUF = Lay<KVF>::NPBUF;
    const uint32_t pempty_r = ptx::mapa(bar_addr<KVF>(base, B_PEMPTY), 0);  // the score CTA's barriers
    uint32_t g = 0;
    Segment sg;
    while (c.next(a.qs, &sg)) {
        for (int pg = sg.page_begin; pg < sg.page_end; ++pg, ++g) {
            if (!warp_wait(bar_addr<KVF>(base, B_PVDONE + g % NPBUF), (g / NPBUF) & 1u, wc, false, lane)) return;
            if (lane == 0) ptx::mbar_arrive_remote(pempty_r + 8u * (g % NPBUF));
        }
    }
}

template <int KVF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Lay<KVF>::NTHREADS, 1)
    tc_attention_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmq,
                        const TcArgs args) {
    using L = Lay<KVF>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const AttnArgs& a = args.a;
    const uint32_t base = ptx::smem_u32(smem);
    if (base & 1023u) {  // both CTAs share the layout, so both leave here together
        if (threadIdx.x == 0) set_device_error(MLA_ERR_UNSUPPORTED);
        return;
    }
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    long long* red = reinterpret_cast<long long*>(smem + L::OFF_RED);

    // the split combine (a programmatic dependent) may be scheduled now; it waits for this
    // grid's completion before it reads anything this kernel writes
    launch_dependents();
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int unit = blockIdx.x >> 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Set-up runs side by side: warp 2 initialises the barriers, warp 1 allocates TMEM, and
    // warp 0 computes the split schedule (its loads of the sequence lengths are the long pole).
    if (threadIdx.x == 64) {
        for (int s = 0; s < (L::STAGES > L::VSTAGES ? L::STAGES : L::VSTAGES); ++s) {
            // MX caches: the four converter warps complete every stage (a query stage also
            // waits for the TMA's bytes)
            ptx::mbar_init(bar_addr<KVF>(base, B_FULL + s), KVF == KV_PLAIN ? 1 : 4);
            ptx::mbar_init(bar_addr<KVF>(base, B_FULLP + 2 * s), KVF == KV_PLAIN ? 1 : 4);
            ptx::mbar_init(bar_addr<KVF>(base, B_FULLP + 2 * s + 1), KVF == KV_PLAIN ? 1 : 4);
            ptx::mbar_init(bar_addr<KVF>(base, B_EMPTY + s), 1);
        }
        for (int s = 0; s < L::RAW_STAGES; ++s) {
            ptx::mbar_init(bar_addr<KVF>(base, B_RFULL + s), 1);
            ptx::mbar_init(bar_addr<KVF>(base, B_REMPTY + s), 4);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_addr<KVF>(base, B_SFULL + b), 1);
            ptx::mbar_init(bar_addr<KVF>(base, B_SFREE + b), 4);
        }
        for (int b = 0; b < L::NPBUF; ++b) {
            ptx::mbar_init(bar_addr<KVF>(base, B_PFULL + b), 1);
            ptx::mbar_init(bar_addr<KVF>(base, B_PEMPTY + b), 1);
            ptx::mbar_init(bar_addr<KVF>(base, B_PREADY + b), 4);
            ptx::mbar_init(bar_addr<KVF>(base, B_PVDONE + b), 1);
        }
        ptx::mbar_init(bar_addr<KVF>(base, B_OFREE), 4);
        ptx::mbar_init(bar_addr<KVF>(base, B_DONE), rank == 0 ? 2 : 1);  // score CTA: two issuers
        ptx::mbar_init(bar_addr<KVF>(base, B_QREADY), 4);
        ptx::mbar_init(bar_addr<KVF>(base, B_QSEEN), 2);
        ptx::mbar_init(bar_addr<KVF>(base, B_DRYW), 1);
        ptx::mbar_init(bar_addr<KVF>(base, B_DRYC), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmap);
        ptx::prefetch_tmap(&tmq);
    }
    if (warp == 1) {
        ptx::tmem_alloc(base + L::OFF_MISC, 512);
        ptx::tmem_relinquish();
    }
    // Launched as a programmatic dependent, this kernel may start while the kernels before it
    // (the absorption GEMM, and before that possibly a cache append) finish.  Lengths and page
    // table come from earlier work and are read at once; both producers wait for the preceding
    // grid (griddepcontrol.wait) before loading queries or cache rows.
    UnitCursor cur;
    long long per;
    cur.init(a.qs, unit, a.n_units, red, &per);  // ends with a block barrier
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_sync();  // the peer's barriers are initialised before any remote arrive
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{args.wait_ns, abort_flag, false};

    if (warp == 0) {
        if (lane == 0) {
            if (rank == 0) producer<KVF, L::STAGES>(a, &tmap, &tmq, cur, base, rank, wc);
            else producer<KVF, L::VSTAGES>(a, &tmap, &tmq, cur, base, rank, wc);
        }
    } else if (warp == 1) {
        if (rank == 0) score_mma<KVF, 0>(a, cur, base, tmem, wc, lane);
        else value_mma<KVF>(a, cur, base, tmem, wc, lane);
    } else if (warp == 6) {
        if (rank == 1) value_release<KVF>(a, cur, base, lane, wc);
        else score_mma<KVF, 1>(a, cur, base, tmem, wc, lane);
    } else if (warp >= 7) {
        if (KVF != KV_PLAIN) converter<KVF>(a, &tmq, cur, base, rank, warp - 7, lane, wc);
    } else if (rank == 0) {
        score_softmax<KVF>(args, cur, base, tmem, peer, warp, lane, wc);
    } else {
        value_warps<KVF>(a, cur, base, tmem, warp, lane, wc);
    }
    // every CTA waits for the preceding grid before it leaves, even one without work: this
    // grid's completion then implies that grid's, which the combine after it relies on
    if (threadIdx.x == 0) grid_dependency_wait();
    ptx::tc_fence_before();
    __syncthreads();
    if (*abort_flag) {  // give copies that a peer may still have in flight time to land
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) {
        }
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    ptx::cluster_sync();  // no CTA leaves while its peer may still write into it
}

// ----------------------------------------------------------------------------- host side
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D map over rows of 576 bf16 ([num_pages*64 rows, 576 columns]); box 64 columns x box_rows,
// 128-byte swizzle.
inline bool encode_pool_map(CUtensorMap* tm, void* pool, long long num_pages, uint32_t box_rows = 64) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)WID, (cuuint64_t)num_pages * PAGE};
    cuuint64_t strides[1] = {(cuuint64_t)WID * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tca

inline bool tc_attention_supported(const mla_config* c, const mla_cache* k, int cc_major, int cc_minor) {
    return c->dtype == MLA_BF16 && c->n_heads == tca::NH && c->d_latent == tca::DC && c->d_rope == tca::DR &&
           c->page_size == tca::PAGE && cc_major == 10 && cc_minor == 3 && k->num_pages * tca::PAGE < (1LL << 31);
}

template <int KVF>
inline mla_status tc_attention_launch_fmt(const AttnArgs& a, const mla_cache* cache, unsigned long long wait_ns,
                                          bool pdl, cudaStream_t stream) {
    using L = tca::Lay<KVF>;
    CUtensorMap tm, tmq;
    // the query rows viewed as [n_queries * 128, 576] bf16, box 64 columns x 64 rows
    if (!tca::encode_pool_map(&tmq, const_cast<void*>(a.q_cat), (long long)a.qs.n_queries * tca::NH / tca::PAGE))
        return MLA_ERR_CUDA;
    if (KVF == KV_PLAIN) {
        if (!tca::encode_pool_map(&tm, cache->pool, cache->num_pages)) return MLA_ERR_CUDA;
    } else {
        tm = tmq;  // unused: MX pages arrive by plain bulk copies
    }
    tca::TcArgs t;
    t.a = a;
    t.wait_ns = wait_ns;
    t.scale_log2 = a.scale * 1.4426950408889634f;
    if (cudaFuncSetAttribute(tca::tc_attention_kernel<KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::SMEM_BYTES) != cudaSuccess)
        return MLA_ERR_CUDA;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2 * a.n_units);
    lc.blockDim = dim3(L::NTHREADS);
    lc.dynamicSmemBytes = L::SMEM_BYTES;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&lc, tca::tc_attention_kernel<KVF>, tm, tmq, t) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

inline mla_status tc_attention_launch(const AttnArgs& a, const mla_cache* cache, unsigned long long wait_ns,
                                      bool pdl, cudaStream_t stream) {
    switch (cache->kv_format) {
        case MLA_KV_PLAIN: return tc_attention_launch_fmt<KV_PLAIN>(a, cache, wait_ns, pdl, stream);
        case MLA_KV_MXFP8: return tc_attention_launch_fmt<KV_MXFP8>(a, cache, wait_ns, pdl, stream);
        case MLA_KV_MXFP4: return tc_attention_launch_fmt<KV_MXFP4>(a, cache, wait_ns, pdl, stream);
    }
    return MLA_ERR_INVALID_ARG;
}

}  // namespace mla
