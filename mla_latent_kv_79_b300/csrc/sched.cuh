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
//
// Query-aligned variant (decode only): when every query can have at least one unit of its
// own, query q gets k_q = max(1, floor(P_q * U / total)) units, cut into pieces of
// ceil(P_q / k_q) pages, and no unit spans two queries (a unit that would otherwise finish
// one query and start the next pays a second drain and query load).  It is used when it fits
// (sum k_q <= U) and its largest piece is at most 5/4 of the flat `per` (plus one page).
// A split query's piece i writes slot 2 * (K_q + i), K_q = sum of k over the queries before q.
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
    int flat_only;         // 1: never use the query-aligned schedule
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

// Scratch for the block-wide helpers (reduction words and broadcasts).
constexpr int SCHED_SCRATCH = 35;

// Units of query q (with np pages) in the query-aligned schedule.
__device__ __forceinline__ long long aligned_units(int np, int n_units, long long total) {
    if (np <= 0) return 0;
    const long long k = (long long)np * n_units / total;
    return k > 0 ? k : 1;
}

// The schedule of one call, identical in every CTA of the attention kernel and the combine.
struct Plan {
    bool aligned;
    long long total;  // pages of all queries
    long long per;    // flat partition: pages per unit
};





struct Segment {
    int q, seq, len;         // query, its sequence, its visible length
    int page_begin, page_end;
    int n_pages;             // pages of the whole query
    int slot;                // partial slot if split
    bool direct;             // segment covers the whole query
    bool first_of_unit;
};

// ---- one-warp versions (every lane gets the result): the unit cursor's set-up is on the
// critical path of every CTA, so it uses shuffles only, no block barriers.
__device__ __forceinline__ long long warp_sum_ll(long long v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ long long warp_max_ll(long long v) {
    for (int o = 16; o > 0; o >>= 1) {
        const long long t = __shfl_xor_sync(0xffffffffu, v, o);
        v = t > v ? t : v;
    }
    return v;
}

__device__ Plan warp_plan(const QuerySet& qs, int n_units) {
    const int lane = threadIdx.x & 31;
    Plan p;
    if (qs.mode == 1) {
        p.total = ceil_sum(qs.q_start + (long long)qs.n_queries, qs.page_size) - ceil_sum(qs.q_start, qs.page_size);
    } else {
        long long t = 0;
        for (int q = lane; q < qs.n_queries; q += 32) t += query_pages(qs, q);
        p.total = warp_sum_ll(t);
    }
    p.per = (p.total + n_units - 1) / n_units;
    if (p.per < 1) p.per = 1;
    p.aligned = false;
    if (qs.mode != 0 || p.total == 0 || qs.flat_only) return p;
    long long ks = 0, worst = 0;
    for (int q = lane; q < qs.n_queries; q += 32) {
        const int np = query_pages(qs, q);
        const long long k = aligned_units(np, n_units, p.total);
        if (k == 0) continue;
        ks += k;
        const long long pc = (np + k - 1) / k;
        worst = pc > worst ? pc : worst;
    }
    const long long K = warp_sum_ll(ks), W = warp_max_ll(worst);
    p.aligned = K <= n_units && 4 * W <= 5 * p.per + 4;
    return p;
}

// First query q whose inclusive prefix of value(q) exceeds `target`, and target minus the
// prefix before q; q = -1 when the total does not exceed target.  One warp.
template <typename F>
__device__ void warp_find(int n_queries, long long target, F value, int* q_out, long long* off_out) {
    const int lane = threadIdx.x & 31;
    long long run = 0;
    for (int c0 = 0; c0 < n_queries; c0 += 32) {
        const int q = c0 + lane;
        const long long v0 = q < n_queries ? value(q) : 0;
        long long v = v0;
        for (int o = 1; o < 32; o <<= 1) {
            const long long t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        const long long incl = run + v, excl = incl - v0;
        const unsigned hit = __ballot_sync(0xffffffffu, q < n_queries && v0 > 0 && excl <= target && target < incl);
        if (hit) {
            const int src = __ffs(hit) - 1;
            *q_out = c0 + src;
            *off_out = __shfl_sync(0xffffffffu, target - excl, src);
            return;
        }
        run = __shfl_sync(0xffffffffu, incl, 31);
    }
    *q_out = -1;
    *off_out = 0;
}

// The plan for a whole block: warp 0 computes it, red[0..2] carries it to the other warps.
__device__ Plan block_plan(const QuerySet& qs, int n_units, long long* red) {
    if (threadIdx.x < 32) {
        const Plan p = warp_plan(qs, n_units);
        if (threadIdx.x == 0) {
            red[0] = p.aligned;
            red[1] = p.total;
            red[2] = p.per;
        }
    }
    __syncthreads();
    Plan p;
    p.aligned = red[0] != 0;
    p.total = red[1];
    p.per = red[2];
    __syncthreads();
    return p;
}

// Walks the segments of one unit.  Initialised block-wide; next() is thread-uniform.
struct UnitCursor {
    long long flat, flat_end;
    int q, page, unit;
    bool first;
    bool aligned;      // query-aligned schedule: one segment [page, a_end) of query q
    int a_end;

    // Warp 0 computes the plan and the unit's start; the block reads them from red[0..5].
    __device__ void init(const QuerySet& qs, int u, int n_units, long long* red, long long* per_out) {
        if (threadIdx.x < 32) {
            const Plan pl = warp_plan(qs, n_units);
            long long r_flat = 0, r_end = 0, r_q = 0, r_page = 0, r_aend = 0;
            if (pl.aligned) {
                int qq;
                long long piece;
                const long long total = pl.total;
                warp_find(qs.n_queries, (long long)u,
                          [&](int i) { return aligned_units(query_pages(qs, i), n_units, total); }, &qq, &piece);
                if (qq >= 0) {
                    const int np = query_pages(qs, qq);
                    const long long k = aligned_units(np, n_units, total), pc = (np + k - 1) / k, b = piece * pc;
                    if (b < np) {
                        r_q = qq;
                        r_page = b;
                        r_aend = b + pc < np ? b + pc : np;
                        r_end = 1;
                    }
                }
            } else {
                r_flat = (long long)u * pl.per;
                r_end = r_flat + pl.per < pl.total ? r_flat + pl.per : pl.total;
                if (r_flat < r_end) {
                    int qq;
                    long long off;
                    if (qs.mode == 1) {
                        // prefill: page counts follow a closed form; bisect the query
                        int lo = 0, hi = qs.n_queries - 1;
                        const long long base = ceil_sum(qs.q_start, qs.page_size);
                        while (lo < hi) {
                            const int mid = (lo + hi) >> 1;
                            if (ceil_sum(qs.q_start + (long long)mid + 1, qs.page_size) - base > r_flat) hi = mid;
                            else lo = mid + 1;
                        }
                        qq = lo;
                        off = r_flat - (ceil_sum(qs.q_start + (long long)lo, qs.page_size) - base);
                    } else {
                        warp_find(qs.n_queries, r_flat, [&](int i) { return (long long)query_pages(qs, i); }, &qq, &off);
                    }
                    r_q = qq < 0 ? 0 : qq;
                    r_page = off;
                }
            }
            if (threadIdx.x == 0) {
                red[0] = pl.aligned;
                red[1] = pl.per;
                red[2] = r_flat;
                red[3] = r_end;
                red[4] = r_q;
                red[5] = r_page;
                red[6] = r_aend;
            }
        }
        __syncthreads();
        aligned = red[0] != 0;
        *per_out = red[1];
        flat = red[2];
        flat_end = red[3];
        q = (int)red[4];
        page = (int)red[5];
        a_end = (int)red[6];
        unit = u;
        first = true;
        __syncthreads();
    }

    __device__ bool next(const QuerySet& qs, Segment* s) {
        if (aligned) {
            if (flat >= flat_end) return false;
            const int np = query_pages(qs, q);
            s->q = q;
            s->seq = query_seq(qs, q);
            s->len = query_len(qs, q);
            s->page_begin = page;
            s->page_end = a_end;
            s->n_pages = np;
            s->first_of_unit = true;
            s->slot = 2 * unit;
            s->direct = (page == 0 && a_end == np);
            flat = flat_end;
            return true;
        }
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
