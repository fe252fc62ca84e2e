// Portable SIMT GEMM used by mla_cache_append / mla_absorb_q / mla_out for shapes and types
// the tcgen05 kernels do not take (fp32, small or odd dimensions).
//
//   C[m, n] = sum_k A[m, k] * B(k, n)           (fp32 accumulation)
//
// batched over blockIdx.z (the head for absorb/out).  A is row-major with leading dimension
// lda; B(k, n) = B[k*ldb_k + n*ldb_n] so both [K,N] and [N,K] weight views are served.
// Tile 64x64x16, 256 threads, 4x4 outputs per thread.
#pragma once

#include "mla_common.cuh"

namespace mla {

enum SimtEpilogue { EPI_STORE = 0, EPI_APPEND = 1 };

struct SimtGemmArgs {
    const void* A; long long lda, a_batch;
    const void* B; long long ldb_k, ldb_n, b_batch;
    const void* B2; long long ldb2_k;   // append: W_KR for columns n >= n_split
    int n_split;                         // append: d_c (columns >= n_split come from B2)
    void* C; long long ldc, c_batch;     // EPI_STORE: C[m*ldc + n] (+ batch offset)
    int M, N, K;
    // append epilogue
    const int* seq_idx; const int* pos;
    const int* page_table; int max_pages; int batch; int page_size; long long num_pages;
    int width;                           // W (row width of the pool)
    RopeFreq rf;                         // append: frequencies of the RoPE pairs
};

template <typename T, int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemmArgs g) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int z = blockIdx.z;
    const T* A = reinterpret_cast<const T*>(g.A) + (long long)z * g.a_batch;
    const T* B = reinterpret_cast<const T*>(g.B) + (long long)z * g.b_batch;
    const T* B2 = reinterpret_cast<const T*>(g.B2);
    const bool b_n_contig = (g.ldb_n == 1);

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < g.K; k0 += BK) {
        // A tile: 64 rows x 16 k; thread loads 4 elements along k-contiguous rows
        for (int e = tid; e < BM * BK; e += 256) {
            int mm = e / BK, kk = e % BK;
            int m = m0 + mm, k = k0 + kk;
            As[kk][mm] = (m < g.M && k < g.K) ? to_f32(A[(long long)m * g.lda + k]) : 0.f;
        }
        for (int e = tid; e < BM * BK; e += 256) {
            int kk, nn;
            if (b_n_contig) { kk = e / BN; nn = e % BN; } else { nn = e / BK; kk = e % BK; }
            int k = k0 + kk, n = n0 + nn;
            float v = 0.f;
            if (k < g.K && n < g.N) {
                if (EPI == EPI_APPEND && n >= g.n_split)
                    v = to_f32(B2[(long long)k * g.ldb2_k + (n - g.n_split)]);
                else
                    v = to_f32(B[(long long)k * g.ldb_k + (long long)n * g.ldb_n]);
            }
            Bs[kk][nn] = v;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= g.M) continue;
        if (EPI == EPI_STORE) {
            T* C = reinterpret_cast<T*>(g.C) + (long long)z * g.c_batch + (long long)m * g.ldc;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                int n = n0 + tx * 4 + j;
                if (n < g.N) C[n] = from_f32<T>(acc[i][j]);
            }
        } else {
            // append: RoPE on columns >= n_split, then scatter into the paged pool
            const int b = __ldg(g.seq_idx + m), p = __ldg(g.pos + m);
            if (b < 0 || b >= g.batch || p < 0 || p >= g.max_pages * g.page_size) {
                if (tx == 0) set_device_error(MLA_ERR_DEVICE_BOUNDS);
                continue;
            }
            const int page = __ldg(g.page_table + (long long)b * g.max_pages + p / g.page_size);
            if (page < 0 || page >= g.num_pages) {
                if (tx == 0) set_device_error(MLA_ERR_DEVICE_BOUNDS);
                continue;
            }
            T* row = reinterpret_cast<T*>(g.C) +
                     ((long long)page * g.page_size + p % g.page_size) * g.width;
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                int n = n0 + tx * 4 + j;
                float v0 = acc[i][j], v1 = acc[i][j + 1];
                if (n >= g.n_split && n < g.N) {
                    float c, s;
                    rope_cos_sin(p, g.rf.theta[(n - g.n_split) / 2], &c, &s);
                    float r0 = v0 * c - v1 * s, r1 = v0 * s + v1 * c;
                    v0 = r0; v1 = r1;
                }
                if (n < g.N) row[n] = from_f32<T>(v0);
                if (n + 1 < g.N) row[n + 1] = from_f32<T>(v1);
            }
        }
    }
}

// RoPE part of the absorbed query: q_cat[n,h,d_c+2i : d_c+2i+2] = rotate(q_rope[n,h,2i:2i+2], pos[n]).
// Grid (n_tokens, ceil(n_h / ROPE_HEADS)): the d_r/2 (cos, sin) of the token are evaluated once
// per block into shared memory; each thread then rotates a few pairs.
constexpr int ROPE_HEADS = 16;

template <typename T>
__global__ void __launch_bounds__(256) rope_query_kernel(const T* __restrict__ q_rope, const int* __restrict__ pos,
                                                         T* __restrict__ q_cat, int n_tokens, int n_h, int d_r,
                                                         int d_c, const __grid_constant__ RopeFreq rf) {
    __shared__ float cs[512], sn[512];   // d_r <= 1024
    launch_dependents();  // the absorption GEMM writes the other columns of q_cat
    const int n = blockIdx.x;
    const int h0 = blockIdx.y * ROPE_HEADS;
    const int half = d_r / 2;
    const int p = __ldg(pos + n);
    for (int i = threadIdx.x; i < half; i += blockDim.x) rope_cos_sin(p, rf.theta[i], &cs[i], &sn[i]);
    __syncthreads();
    const int nh = min(ROPE_HEADS, n_h - h0);
    for (int e = threadIdx.x; e < nh * half; e += blockDim.x) {
        const int h = h0 + e / half, i = e % half;
        const long long row = (long long)n * n_h + h;
        const T* src = q_rope + row * d_r + 2 * i;
        T* dst = q_cat + row * (long long)(d_c + d_r) + d_c + 2 * i;
        const float x0 = to_f32(src[0]), x1 = to_f32(src[1]);
        dst[0] = from_f32<T>(x0 * cs[i] - x1 * sn[i]);
        dst[1] = from_f32<T>(x0 * sn[i] + x1 * cs[i]);
    }
}

}  // namespace mla
