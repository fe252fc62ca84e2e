// Split-over-length schedule shared by the attention kernels and the combine kernel.
//
// The work of one call is the flat list of (query, page) pairs, queries in order, each query
// owning ceil(len/P) pages.  It is cut into U units of `per` consecutive pages
// (per = ceil(total/U)), one unit per CTA (or CTA pair).  Inside a unit the pages of one
// query form a segment.  A segment that covers its whole query writes the final output
// directly; a split segment writes a partial (o/l, lse) to slot 2u (if it is the unit's
// first segment) or 2u+1 (its last), and the combine kernel merges the partials of every
// split query.  Everything is recomputed on the device from seq_lens, so a call needs no
// host-side view of the lengths and no planning buffer.
#pragma once

#include "mla_common.cuh"

namespace mla {

struct QuerySet {
    int mode;              // 0: decode (query q is sequence q); 1: prefill (queries of one sequence)
    int n_queries;
    const int* seq_lens;   // decode: visible length of query q
    int seq;               // prefill: the sequence
    int q_start;           // prefill: position of query 0 (query i sees t <= q_start + i)
    int page_size;
    int max_len;           // max_pages * page_size
};

__device__ __forceinline__ int query_seq(const QuerySet& qs, int q) { return qs.mode == 0 ? q : qs.seq; }

__device__ __forceinline__ int query_len(const QuerySet& qs, int q) {
    int len = qs.mode == 0 ? __ldg(qs.seq_lens + q) : qs.q_start + q + 1;
    if (len < 0) { set_device_error(MLA_ERR_DEVICE_BOUNDS); len = 0; }
    if (len > qs.max_len) { set_device_error(MLA_ERR_DEVICE_BOUNDS); len = qs.max_len; }
    return len;
}

__device__ __forceinline__ int query_pages(const QuerySet& qs, int q) {
    return (query_len(qs, q) + qs.page_size - 1) / qs.page_size;
}

// sum_{m=1..n} ceil(m / P)
__device__ __forceinline__ long long ceil_sum(long long n, int P) {
    long long k = n / P, r = n % P;
    return (long long)P * k * (k + 1) / 2 + r * (k + 1);
}

// Block-wide sum of a long long (every thread gets the result).  Uses 33 words of smem.
__device__ __forceinline__ long long block_sum_ll(long long v, long long* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        long long s = 0;
        for (int i = 0; i < nw; ++i) s += red[i];
        red[32] = s;
    }
    __syncthreads();
    return red[32];
}

// Pages of queries [0, q) (P_q).  Block-wide.
__device__ long long block_prefix_pages(const QuerySet& qs, int q, long long* red) {
    if (qs.mode == 1) return ceil_sum(qs.q_start + (long long)q, qs.page_size) - ceil_sum(qs.q_start, qs.page_size);
    long long s = 0;
    for (int i = threadIdx.x; i < q; i += blockDim.x) s += query_pages(qs, i);
    return block_sum_ll(s, red);
}

// Scratch for the block-wide helpers: red[0..32] reduction words, red[33..34] locate result.
constexpr int SCHED_SCRATCH = 35;

// First query q with P_{q+1} > flat, and the page offset of `flat` inside it.  Block-wide.
// `flat` must be < total.
__device__ void block_locate(const QuerySet& qs, long long flat, int* q_out, int* page_out, long long* red) {
    if (qs.mode == 1) {
        int lo = 0, hi = qs.n_queries - 1;
        long long base = ceil_sum(qs.q_start, qs.page_size);
        while (lo < hi) {  // smallest q with P_{q+1} > flat
            int mid = (lo + hi) >> 1;
            long long p_next = ceil_sum(qs.q_start + (long long)mid + 1, qs.page_size) - base;
            if (p_next > flat) hi = mid; else lo = mid + 1;
        }
        long long p_q = ceil_sum(qs.q_start + (long long)lo, qs.page_size) - base;
        *q_out = lo;
        *page_out = (int)(flat - p_q);
        return;
    }
    // decode: stream the lengths in chunks of blockDim with a running offset.
    long long& s_found_q = red[33];
    long long& s_found_page = red[34];
    if (threadIdx.x == 0) { s_found_q = -1; s_found_page = 0; }
    long long run = 0;
    for (int c0 = 0; c0 < qs.n_queries; c0 += blockDim.x) {
        int q = c0 + threadIdx.x;
        int np = q < qs.n_queries ? query_pages(qs, q) : 0;
        // inclusive scan of np within the block
        long long v = np;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
        for (int o = 1; o < 32; o <<= 1) {
            long long t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        __syncthreads();
        if (lane == 31) red[warp] = v;
        __syncthreads();
        long long warp_off = 0;
        for (int i = 0; i < warp; ++i) warp_off += red[i];
        long long incl = run + warp_off + v;   // P_{q+1}
        long long excl = incl - np;            // P_q
        if (q < qs.n_queries && np > 0 && excl <= flat && flat < incl) {
            s_found_q = q;
            s_found_page = (int)(flat - excl);
        }
        long long chunk = 0;
        for (int i = 0; i < nw; ++i) chunk += red[i];
        __syncthreads();
        run += chunk;
        if (s_found_q >= 0) break;  // uniform: read after the barrier
    }
    __syncthreads();
    *q_out = s_found_q < 0 ? 0 : (int)s_found_q;
    *page_out = (int)s_found_page;
    __syncthreads();
}

__device__ __forceinline__ long long block_total_pages(const QuerySet& qs, long long* red) {
    return block_prefix_pages(qs, qs.n_queries, red);
}

struct Segment {
    int q, seq, len;         // query, its sequence, its visible length
    int page_begin, page_end;
    int n_pages;             // pages of the whole query
    int slot;                // partial slot if split
    bool direct;             // segment covers the whole query
    bool first_of_unit;
};

// Walks the segments of one unit.  Initialised block-wide; next() is thread-uniform.
struct UnitCursor {
    long long flat, flat_end;
    int q, page, unit;
    bool first;

    __device__ void init(const QuerySet& qs, int u, int n_units, long long* red, long long* per_out) {
        long long total = block_total_pages(qs, red);
        long long per = (total + n_units - 1) / n_units;
        if (per < 1) per = 1;
        *per_out = per;
        unit = u;
        flat = (long long)u * per;
        flat_end = flat + per < total ? flat + per : total;
        first = true;
        q = 0; page = 0;
        if (flat < flat_end) block_locate(qs, flat, &q, &page, red);
    }

    __device__ bool next(const QuerySet& qs, Segment* s) {
        if (flat >= flat_end) return false;
        int np = query_pages(qs, q);
        while (np == 0 && q + 1 < qs.n_queries) { ++q; page = 0; np = query_pages(qs, q); }
        if (np == 0) { flat = flat_end; return false; }
        long long left = flat_end - flat;
        int take = (int)((long long)(np - page) < left ? (long long)(np - page) : left);
        s->q = q;
        s->seq = query_seq(qs, q);
        s->len = query_len(qs, q);
        s->page_begin = page;
        s->page_end = page + take;
        s->n_pages = np;
        s->first_of_unit = first;
        s->slot = first ? 2 * unit : 2 * unit + 1;
        s->direct = (page == 0 && take == np);
        flat += take;
        page += take;
        if (page == np) { ++q; page = 0; }
        first = false;
        return true;
    }
};

}  // namespace mla
