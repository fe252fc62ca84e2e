// Portable SIMT split attention over the paged latent cache (any dimensions, fp32 or bf16).
//
// Grid (U units, ceil(n_h/HG) head groups), 256 threads.  Each CTA walks the segments of its
// unit (see sched.cuh); for each block of TB tokens it stages the cached rows in shared
// memory as fp32, forms the HG x TB scores, updates the running max / sum per head (online
// softmax) and accumulates o[h, :] += p[h, t] * c_kv[t, :].
#pragma once

#include "mx_format.cuh"
#include "sched.cuh"

namespace mla {

struct AttnArgs {
    QuerySet qs;
    const void* q_cat;          // [Q, n_h, W]
    const void* pool;           // [num_pages, P, W] elements, or the codes of an MX cache
    const void* scales;         // MX cache: [num_pages, P, W / 32] E8M0 scale bytes
    const int* page_table;      // [batch, max_pages]
    int max_pages;
    long long num_pages;
    void* o_lat;                // [Q, n_h, d_c] final output (dtype)
    float* lse;                 // [Q, n_h]
    void* part_o;               // [2U, d_c/V, n_h, V] partials (o / l) of the output dtype, see part_index
    float* part_lse;            // [2U, n_h]
    int n_units;
    int n_h, d_c, width;
    float scale;
};

constexpr int SIMT_TB = 32;     // tokens per staged block

// Split partials are stored in the output dtype T, head-contiguous per 16-byte column group:
// [slot][c/V][h][c%V] with V = 16 / sizeof(T), so that a warp of consecutive heads writes (and
// the combine reads) contiguous memory.  d_c is a multiple of 8.
template <typename T>
__device__ __forceinline__ size_t part_index(long long slot, int h, int c, int n_h, int d_c) {
    constexpr int V = 16 / sizeof(T);
    return (((size_t)slot * (d_c / V) + (c / V)) * n_h + h) * V + (c % V);
}

__host__ __device__ inline size_t simt_attn_smem_bytes(int hg, int width, int d_c) {
    return sizeof(float) * ((size_t)hg * (width + 1) + (size_t)SIMT_TB * (width + 1) +
                            (size_t)hg * SIMT_TB + (size_t)hg * d_c + 3 * (size_t)hg);
}

// KVF: the cache's element format (KV_PLAIN rows of T, or an MX cache read as its dequantised
// values).
template <typename T, int KVF>
__global__ void __launch_bounds__(256) simt_attention_kernel(AttnArgs a, int hg) {
    extern __shared__ float smem[];
    __shared__ long long red[SCHED_SCRATCH];
    const int W = a.width, Wp = W + 1, d_c = a.d_c;
    float* q_s = smem;                           // [hg][Wp]
    float* rows = q_s + (size_t)hg * Wp;         // [TB][Wp]
    float* P = rows + (size_t)SIMT_TB * Wp;      // [hg][TB]
    float* acc = P + (size_t)hg * SIMT_TB;       // [hg][d_c]
    float* m_s = acc + (size_t)hg * d_c;         // [hg]
    float* l_s = m_s + hg;                       // [hg]
    float* alpha_s = l_s + hg;                   // [hg]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int h0 = blockIdx.y * hg;
    const int nh_here = min(hg, a.n_h - h0);
    const T* qc = reinterpret_cast<const T*>(a.q_cat);
    const T* pool = reinterpret_cast<const T*>(a.pool);
    const int ps = a.qs.page_size;

    UnitCursor cur;
    long long per;
    cur.init(a.qs, blockIdx.x, a.n_units, red, &per);
    Segment sg;
    while (cur.next(a.qs, &sg)) {
        // stage the queries of this head group, reset the running state
        for (int e = tid; e < hg * W; e += blockDim.x) {
            int h = e / W, k = e % W;
            q_s[h * Wp + k] = h < nh_here ? to_f32(qc[((long long)sg.q * a.n_h + h0 + h) * W + k]) : 0.f;
        }
        for (int e = tid; e < hg * d_c; e += blockDim.x) acc[e] = 0.f;
        for (int h = tid; h < hg; h += blockDim.x) { m_s[h] = -INFINITY; l_s[h] = 0.f; }
        __syncthreads();

        const int t_begin = sg.page_begin * ps;
        const int t_end = min(sg.page_end * ps, sg.len);
        for (int t0 = t_begin; t0 < t_end; t0 += SIMT_TB) {
            // stage TB rows (token order), masking invalid pages
            for (int e = tid; e < SIMT_TB * W; e += blockDim.x) {
                int j = e / W, k = e % W, t = t0 + j;
                float v = 0.f;
                if (t < t_end) {
                    int page = __ldg(a.page_table + (long long)sg.seq * a.max_pages + t / ps);
                    if (page >= 0 && page < a.num_pages) {
                        const long long row = (long long)page * ps + t % ps;
                        if (KVF == KV_PLAIN)
                            v = to_f32(pool[row * W + k]);
                        else
                            v = mx_load<KVF>(reinterpret_cast<const uint8_t*>(a.pool) + row * mx_row_bytes(KVF, W),
                                             reinterpret_cast<const uint8_t*>(a.scales) + row * mx_scale_bytes(W), k);
                    }
                    else if (k == 0)
                        set_device_error(MLA_ERR_DEVICE_BOUNDS);
                }
                rows[j * Wp + k] = v;
            }
            __syncthreads();
            // scores
            for (int e = tid; e < hg * SIMT_TB; e += blockDim.x) {
                int h = e / SIMT_TB, j = e % SIMT_TB, t = t0 + j;
                float s = -INFINITY;
                if (h < nh_here && t < t_end) {
                    const float* qr = q_s + h * Wp;
                    const float* rr = rows + j * Wp;
                    float d = 0.f;
                    for (int k = 0; k < W; ++k) d = fmaf(qr[k], rr[k], d);
                    s = d * a.scale;
                }
                P[h * SIMT_TB + j] = s;
            }
            __syncthreads();
            // online softmax update, one warp per head
            for (int h = warp; h < hg; h += nwarps) {
                float s0 = P[h * SIMT_TB + lane];
                float mx = warp_max(s0);
                float m_old = m_s[h];
                float m_new = fmaxf(m_old, mx);
                float p0 = 0.f, alpha = 1.f;
                if (m_new != -INFINITY) {
                    p0 = (s0 == -INFINITY) ? 0.f : expf(s0 - m_new);
                    alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
                }
                float sum = warp_sum(p0);
                P[h * SIMT_TB + lane] = p0;
                if (lane == 0) {
                    l_s[h] = l_s[h] * alpha + sum;
                    m_s[h] = m_new;
                    alpha_s[h] = alpha;
                }
            }
            __syncthreads();
            // o += p * c_kv
            for (int e = tid; e < hg * d_c; e += blockDim.x) {
                int h = e / d_c, c = e % d_c;
                float v = acc[e] * alpha_s[h];
                const float* ph = P + h * SIMT_TB;
#pragma unroll 8
                for (int j = 0; j < SIMT_TB; ++j) v = fmaf(ph[j], rows[j * Wp + c], v);
                acc[e] = v;
            }
            __syncthreads();
        }

        // epilogue: final output or split partial
        for (int e = tid; e < nh_here * d_c; e += blockDim.x) {
            int h = e / d_c, c = e % d_c;
            float l = l_s[h];
            float v = l > 0.f ? acc[h * d_c + c] / l : 0.f;
            if (sg.direct)
                reinterpret_cast<T*>(a.o_lat)[((long long)sg.q * a.n_h + h0 + h) * d_c + c] = from_f32<T>(v);
            else
                reinterpret_cast<T*>(a.part_o)[part_index<T>(sg.slot, h0 + h, c, a.n_h, d_c)] = from_f32<T>(v);
        }
        for (int h = tid; h < nh_here; h += blockDim.x) {
            float l = l_s[h];
            float L = l > 0.f ? m_s[h] + logf(l) : -INFINITY;
            if (sg.direct) a.lse[(long long)sg.q * a.n_h + h0 + h] = L;
            else a.part_lse[(long long)sg.slot * a.n_h + h0 + h] = L;
        }
        __syncthreads();
    }
}

// Log-sum-exp merge of the split partials of every split query; also writes the empty-query
// result (o = 0, lse = -inf).  Grid (Q, ceil(n_h * d_c/V / COMBINE_THREADS)): one thread per
// (head, 16-byte column group of V values), heads fastest, so a warp reads 512 contiguous
// bytes of a partial.  The slots of a query are read in batches of COMBINE_BATCH independent
// loads with an online max, i.e. one memory round trip per batch.  The schedule arithmetic
// reads only seq_lens, which the attention kernel does not write, so it runs before the
// grid-dependency wait: launched as a programmatic dependent, it overlaps the attention
// kernel's tail.  Every thread then waits for the attention grid before it stores anything or
// leaves: o_lat and lse may still be read by an earlier kernel of the stream (the previous
// step's output projection) until then, and the kernel after this one (which waits only for
// this grid) must find the attention kernel's direct outputs complete.
constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_BATCH = 8;

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* f) {
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y); f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    } else {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float* f) {
    uint4 u;
    if constexpr (sizeof(T) == 4) {
        u.x = __float_as_uint(f[0]); u.y = __float_as_uint(f[1]); u.z = __float_as_uint(f[2]); u.w = __float_as_uint(f[3]);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&v);
        }
        u.x = w[0]; u.y = w[1]; u.z = w[2]; u.w = w[3];
    }
    return u;
}

template <typename T>
__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(AttnArgs a) {
    constexpr int V = 16 / sizeof(T);
    __shared__ long long red[SCHED_SCRATCH];
    launch_dependents();  // the output projection may stage its weights meanwhile
    const int q = blockIdx.x;
    const int n_h = a.n_h, d_c = a.d_c;
    const int np = query_pages(a.qs, q);
    // the partial slots of query q, as the attention kernel's schedule assigned them: partial i
    // is in slot sbase + 2i, except that in the flat partition the first one is in slot
    // 2*u_lo + 1 when the query starts after the beginning of unit u_lo (its second segment)
    const Plan pl = block_plan(a.qs, a.n_units, red);
    int ns = 0, sbase = 0, first_adj = 0;
    if (pl.aligned) {
        long long kb = 0;
        for (int i = threadIdx.x; i < q; i += blockDim.x) kb += aligned_units(query_pages(a.qs, i), a.n_units, pl.total);
        sbase = (int)(2 * block_sum_ll(kb, red));
        if (np > 0) {
            const long long k = aligned_units(np, a.n_units, pl.total), pc = (np + k - 1) / k;
            ns = (int)((np + pc - 1) / pc);  // non-empty pieces
        }
    } else {
        const long long pq = block_prefix_pages(a.qs, q, red), per = pl.per;
        const long long u_lo = pq / per;
        if (np > 0) ns = (int)((pq + np - 1) / per - u_lo + 1);
        sbase = (int)(2 * u_lo);
        first_adj = pq == u_lo * per ? 0 : 1;
    }
    grid_dependency_wait();  // the attention grid is complete and its writes are visible
    if (np > 0 && ns == 1) return;  // written directly by the attention kernel

    const int e = blockIdx.y * blockDim.x + threadIdx.x;
    if (e >= n_h * (d_c / V)) return;
    const int h = e % n_h, grp = e / n_h;
    uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.o_lat) + ((long long)q * n_h + h) * d_c + V * grp);
    if (np == 0) {
        *out = make_uint4(0u, 0u, 0u, 0u);
        if (grp == 0) a.lse[(long long)q * n_h + h] = -INFINITY;
        return;
    }

    float mx = -INFINITY, wsum = 0.f;
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
    const T* po = reinterpret_cast<const T*>(a.part_o);
    for (int i0 = 0; i0 < ns; i0 += COMBINE_BATCH) {
        float lv[COMBINE_BATCH];
        uint4 v[COMBINE_BATCH];
#pragma unroll
        for (int j = 0; j < COMBINE_BATCH; ++j) {
            lv[j] = -INFINITY;
            v[j] = make_uint4(0u, 0u, 0u, 0u);
            if (i0 + j < ns) {
                const long long sl = sbase + 2 * (i0 + j) + (i0 + j == 0 ? first_adj : 0);
                lv[j] = a.part_lse[sl * n_h + h];
                v[j] = *reinterpret_cast<const uint4*>(po + part_index<T>(sl, h, V * grp, n_h, d_c));
            }
        }
        float m_new = mx;
#pragma unroll
        for (int j = 0; j < COMBINE_BATCH; ++j) m_new = fmaxf(m_new, lv[j]);
        if (m_new == -INFINITY) continue;
        const float r = (mx == -INFINITY) ? 0.f : __expf(mx - m_new);
        wsum *= r;
#pragma unroll
        for (int c = 0; c < V; ++c) acc[c] *= r;
#pragma unroll
        for (int j = 0; j < COMBINE_BATCH; ++j) {
            const float w = (lv[j] == -INFINITY) ? 0.f : __expf(lv[j] - m_new);
            wsum += w;
            float f[V];
            unpack16<T>(v[j], f);
#pragma unroll
            for (int c = 0; c < V; ++c) acc[c] = fmaf(w, f[c], acc[c]);
        }
        mx = m_new;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int c = 0; c < V; ++c) acc[c] *= inv;
    *out = pack16<T>(acc);
    if (grp == 0) a.lse[(long long)q * n_h + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

}  // namespace mla
