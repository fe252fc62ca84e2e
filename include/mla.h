/*
 * mla.h - C ABI of libmla: the data-parallel hot path of Multi-head Latent Attention (MLA)
 * over a paged latent KV cache, for NVIDIA B300 (sm_103a).
 *
 * Sources (page title, section):
 *   [OPN] "Operator Notes (1): MLA - Multi-head Latent Attention at the Operator Level",
 *         section 2 (weight shapes W_DKV [d_model,d_c], W_UK/W_UV [d_c,n_h*d_h],
 *         the chain c_kv = x W_DKV, K = c_kv W_UK, V = c_kv W_UV, softmax(Q K^T/sqrt d) V),
 *         section 3 (only c_kv enters the cache).
 *   [GLO] "multi-head latent attention" glossary: a small decoupled RoPE key is cached beside
 *         the latent; the up-projections are absorbed into the query and output projections;
 *         MLA pairs with PagedAttention.
 *   [RMJ] "Multi-Head Latent Attention and the Compression of the KV Cache": by associativity
 *         the up-projection is absorbed into the query, so attention runs on the latent.
 *   [IPM] "Multi-Head Latent Attention (MLA) Explained": MXFP4 quantisation of the KV cache
 *         (section "Which Models Use MLA and What Is Next").
 *
 * Notation: n_h heads, d_h (= d_nope) per-head width, d_r (= d_rope) RoPE width, d_c latent
 * width, W = d_c + d_r numbers cached per token, P = page_size tokens per page.
 *
 * Conventions that hold for every entry point:
 *   - Every pointer named "device" is CUDA device memory owned by the caller; the library
 *     never allocates, frees or retains it.  Host pointers are read before the call returns.
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).  The returned status
 *     covers host-side argument checks and launch errors only.  Faults found on the device
 *     (a page id outside the pool, a position beyond the page table, a bounded wait that ran
 *     out) are recorded in a per-device error word and read with mla_get_device_error().
 *   - Element type of every floating-point tensor is cfg->dtype (MLA_F32 or MLA_BF16), except
 *     lse, which is always float32.  bf16 is stored as IEEE bfloat16 bits.
 *   - Every tensor pointer must be 16-byte aligned; tensors are dense row-major with the
 *     shapes given below (no strides).
 *   - RoPE rotates interleaved pairs (2i, 2i+1) by pos * rope_base^(-2i/d_r); positions are
 *     0-based.  The score scale is cfg->softmax_scale, or 1/sqrt(d_h + d_r) when it is 0.
 *   - Slots of a plain pool that no token owns must hold finite values (masked tokens still
 *     meet a zero weight: 0 * finite = 0).  An MX cache has no such rule.
 *   - lse is the natural-log log-sum-exp of the scaled scores of one (query, head).
 *   - Kernels are launched with programmatic dependent launch: a kernel of this library may
 *     start while the kernel before it in the stream finishes, if that kernel allows it
 *     (griddepcontrol.launch_dependents; the library's own kernels do).  It waits for that
 *     kernel before reading what that kernel may write: q_cat and the cache rows in
 *     mla_decode / mla_prefill (written by mla_absorb_q and mla_cache_append), o_lat in
 *     mla_out, o in mla_out_proj, x in mla_query_proj, q_nope / q_rope / pos and x in
 *     mla_absorb_q and mla_cache_append.  The page
 *     table and lengths are read without the wait, so they must be produced
 *     by work that completes before the preceding kernel starts (ordinary kernels and copies
 *     do; MLA_TUNE_NO_PDL turns programmatic launch off).
 *
 * Error behaviour: a non-OK status means nothing was launched, except MLA_ERR_CUDA, which
 * reports the CUDA error of a launch (cudaGetLastError is cleared).
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

typedef struct CUstream_st* mla_stream_t; /* a cudaStream_t */

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size or dimension          */
    MLA_ERR_UNSUPPORTED = 2,    /* dimensions the library does not handle                   */
    MLA_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed                     */
    MLA_ERR_WORKSPACE = 4,      /* workspace missing or smaller than the size query returned */
    MLA_ERR_DEVICE_TIMEOUT = 5, /* a device-side bounded wait ran out (device error word)   */
    MLA_ERR_DEVICE_BOUNDS = 6,  /* a page id / position outside the cache (device error word) */
    MLA_ERR_SCRATCH_LIMIT = 7   /* mla_decode_static: the split scratch this configuration needs
                                   on this device exceeds MLA_STATIC_SCRATCH_BYTES             */
} mla_status;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype;

/* Model dimensions ([OPN] section 2 conventions, plus the decoupled RoPE width of [GLO]). */
typedef struct {
    int32_t n_heads;       /* n_h                                   */
    int32_t d_nope;        /* d_h: per-head query/key width without RoPE */
    int32_t d_rope;        /* d_r: width of the decoupled RoPE key (even) */
    int32_t d_latent;      /* d_c: latent width, the cached c_kv      */
    int32_t d_model;       /* hidden width of x                       */
    int32_t page_size;     /* P: tokens per cache page                */
    float rope_base;       /* RoPE base, e.g. 10000                   */
    float softmax_scale;   /* 0 => 1/sqrt(d_nope + d_rope)            */
    int32_t dtype;         /* mla_dtype                               */
} mla_config;

/* Element format of the cached rows.
 * MLA_KV_PLAIN: rows of cfg->dtype numbers.
 * MLA_KV_MXFP8 / MLA_KV_MXFP4: the low-precision cache that [IPM] names (MXFP4 quantisation
 *   of the KV cache), in the block formats of the OCP Microscaling (MX) specification v1.0.
 *   A row of W numbers is cut into W/32 blocks of 32 consecutive elements; each block has one
 *   E8M0 scale byte s (the power of two 2^(s-127)) and 32 element codes, E4M3 bytes (MXFP8)
 *   or E2M1 nibbles (MXFP4; element 2i in the low nibble of byte i).  Element i of block k
 *   of a row stands for 2^(s_k - 127) * value(code_i).  W must be a multiple of 32.
 *   mla_cache_append encodes: block exponent e = the smallest integer with
 *   max|v| <= max_elem * 2^e (max_elem 448 for E4M3, 6 for E2M1), clamped to [-127, 127];
 *   codes round v * 2^-e to nearest, ties to even (the fp32 row after RoPE is the input).
 *   Unlike a plain cache, slots that no token owns may hold any bytes.
 *   [IPM] "Multi-Head Latent Attention (MLA) Explained: What DeepSeek's Architecture Means
 *         for AI Inference Costs", section "Which Models Use MLA and What Is Next". */
typedef enum { MLA_KV_PLAIN = 0, MLA_KV_MXFP8 = 1, MLA_KV_MXFP4 = 2 } mla_kv_format;

/* Paged latent cache ([GLO]: MLA pairs with PagedAttention; [OPN] s.3: only c_kv is cached,
 * here with the RoPE key beside it).  Token t of sequence b lives in row
 * pool[page_table[b*max_pages + t/P]][t%P][0:W]: columns [0,d_c) hold c_kv, [d_c,W) the
 * rotated RoPE key. */
typedef struct {
    void* pool;                 /* device [num_pages, P, W] of cfg->dtype (MLA_KV_PLAIN), or
                                   the codes: [num_pages, P, W] bytes (MXFP8),
                                   [num_pages, P, W/2] bytes (MXFP4)                    */
    int64_t num_pages;
    const int32_t* page_table;  /* device [batch, max_pages] physical page ids         */
    int32_t max_pages;
    int32_t batch;
    const int32_t* seq_lens;    /* device [batch]: cached tokens of each sequence       */
    int32_t kv_format;          /* mla_kv_format (0 for a plain cache)                  */
    void* kv_scales;            /* MX formats: device [num_pages, P, W/32] scale bytes,
                                   16-byte aligned; unused (may be NULL) for a plain cache */
} mla_cache;

/* Build identification: returns MLA_ABI_VERSION. */
#define MLA_ABI_VERSION 2
MLA_API int32_t mla_abi_version(void);

/* Short English text for a status code (static storage). */
MLA_API const char* mla_status_string(mla_status status);

/* mla_cache_append - write new tokens into the latent cache.
 * [OPN] s.2 "c_kv = x @ W_DKV" (the only KV state cached) and [GLO] decoupled RoPE key:
 *   row = [ x[n] @ W_DKV | RoPE(x[n] @ W_KR, pos[n]) ]   (fp32 accumulation, rounded to dtype)
 *   stored to pool[page_table[seq_idx[n]][pos[n]/P]][pos[n]%P].
 * x       device [n_tokens, d_model]
 * w_dkv   device [d_model, d_c]       w_kr device [d_model, d_r]
 * seq_idx device int32 [n_tokens]     pos  device int32 [n_tokens]
 * An MX cache (cache->kv_format) receives the row's codes and block scale bytes instead; that
 * needs cfg->dtype == MLA_BF16 and the tensor-core path (n_h = 128, d_c = 512, d_r = 64, d_model
 * a multiple of 64 on sm_103; else MLA_ERR_UNSUPPORTED).
 * Tokens must target distinct rows.  seq_lens is not modified (the caller owns lengths).
 * A seq_idx outside [0,batch), a position outside the page table or a page id outside the
 * pool sets MLA_ERR_DEVICE_BOUNDS and that token is skipped.  n_tokens == 0 is a no-op. */
MLA_API mla_status mla_cache_append(const mla_config* cfg, const mla_cache* cache, const void* x,
                            const void* w_dkv, const void* w_kr, const int32_t* seq_idx,
                            const int32_t* pos, int32_t n_tokens, mla_stream_t stream);

/* mla_absorb_q - absorbed query ([GLO] absorption paragraph, [RMJ] associativity):
 *   q_cat[n,h,0:d_c]  = q_nope[n,h,:] @ W_UK[:, h*d_h:(h+1)*d_h]^T
 *   q_cat[n,h,d_c:W]  = RoPE(q_rope[n,h,:], pos[n])
 * q_nope device [n_tokens, n_h, d_h]   q_rope device [n_tokens, n_h, d_r] (not rotated)
 * pos    device int32 [n_tokens]       w_uk   device [d_c, n_h*d_h]
 * q_cat  device [n_tokens, n_h, W] (output).  n_tokens == 0 is a no-op. */
MLA_API mla_status mla_absorb_q(const mla_config* cfg, const void* q_nope, const void* q_rope,
                        const int32_t* pos, const void* w_uk, void* q_cat, int32_t n_tokens,
                        mla_stream_t stream);

/* Bytes of device workspace that mla_decode / mla_prefill need on the current device for
 * this configuration (split partials).  The same buffer serves both and may be reused by
 * calls that do not overlap in time. */
MLA_API mla_status mla_workspace_size(const mla_config* cfg, size_t* bytes);

/* mla_decode - one query token per sequence over its whole cached prefix ([OPN] s.2 scores,
 * softmax, weighted sum, in the absorbed form of [GLO]/[RMJ]):
 *   s[b,h,t]  = (q_cat[b,h,:] . pool_row(b,t)) * scale         for t < seq_lens[b]
 *   lse[b,h]  = log sum_t exp(s[b,h,t])
 *   o_lat[b,h,:] = sum_t exp(s[b,h,t] - lse[b,h]) * pool_row(b,t)[0:d_c]
 * q_cat device [batch, n_h, W]; o_lat device [batch, n_h, d_c]; lse device float [batch, n_h].
 * The work is split over the sequence length and merged by a log-sum-exp combine.
 * A sequence with seq_lens[b] == 0 yields o_lat = 0 and lse = -inf.
 * An MX cache is read as its dequantised rows (exactly: every dequantised value is a bf16 number
 * in the range the scales of real data give), so the formulas above hold with pool_row the
 * dequantised row.
 * workspace: device, at least mla_workspace_size() bytes (else MLA_ERR_WORKSPACE). */
MLA_API mla_status mla_decode(const mla_config* cfg, const mla_cache* cache, const void* q_cat,
                      void* o_lat, float* lse, void* workspace, size_t workspace_bytes,
                      mla_stream_t stream);

/* mla_decode_static - mla_decode that allocates nothing and takes no workspace.  The pages
 * have no counterpart: this is a calling convention, not a step of the method.  It serves
 * callers that cannot hand in device memory per call, e.g. a plain C host program with no
 * device allocator of its own, or a serving loop that must not call cudaMalloc / cudaFree
 * (which may synchronise the device) between steps.
 * The split partials go to one fixed array of MLA_STATIC_SCRATCH_BYTES (80 MiB) per device,
 * part of the library's device image: enough for 128 heads x 512 latent columns on up to
 * 159 SMs.  A configuration that needs more (mla_workspace_size() > the limit) is rejected
 * with MLA_ERR_SCRATCH_LIMIT before anything is launched.
 * The first call on each device is its set-up: it looks up that array's address (with the
 * device current), and the driver may place the array in device memory at that moment (lazy
 * module loading).  Make that first call before any stream capture begins; the calls after
 * it allocate nothing.  Nothing in the array has to start
 * at zero: every partial the combine reads is written earlier in the same call.
 * Calls that overlap in time (other streams, other host threads, or an overlapping
 * mla_decode_static on the same device) race on the one array: order them, e.g. on one stream.
 * Arguments, outputs and the other errors are those of mla_decode. */
#define MLA_STATIC_SCRATCH_BYTES ((size_t)80 << 20)
MLA_API mla_status mla_decode_static(const mla_config* cfg, const mla_cache* cache,
                                     const void* q_cat, void* o_lat, float* lse,
                                     mla_stream_t stream);

/* mla_prefill - causal attention of n_queries consecutive tokens of sequence `seq` against
 * that sequence's cache ([OPN] s.2 prefill chain with the causal mask of autoregressive
 * attention): query i sits at position q_start + i and sees tokens t <= q_start + i, which
 * must already be in the cache (append first).  Same formulas and outputs as mla_decode:
 * q_cat device [n_queries, n_h, W]; o_lat device [n_queries, n_h, d_c];
 * lse device float [n_queries, n_h]; workspace as for mla_decode. */
MLA_API mla_status mla_prefill(const mla_config* cfg, const mla_cache* cache, int32_t seq,
                       int32_t q_start, int32_t n_queries, const void* q_cat, void* o_lat,
                       float* lse, void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* mla_prefill_unabsorbed - the prefill chain of [OPN] s.2 in its own form, not absorbed:
 * "Restore K, V from c_kv" (K = c_kv @ W_UK, V = c_kv @ W_UV, every head), then standard
 * causal attention with [GLO]'s decoupled RoPE key, for n_queries consecutive tokens of
 * sequence `seq` (query i at position q_start + i, seeing tokens t <= q_start + i, which must
 * already be in the cache):
 *   s[i,h,t] = ([q_nope[i,h] | RoPE(q_rope[i,h], q_start+i)] . [K[t,h] | k_rope[t]]) * scale
 *   lse[i,h] = log sum_t exp(s[i,h,t])
 *   o[i, h*d_h:(h+1)*d_h] = sum_t exp(s[i,h,t] - lse[i,h]) * V[t,h]
 * This is the same o as mla_prefill followed by mla_out, computed with fewer FLOPs for long
 * prefills (restoring K and V costs 4 L d_c n_h d_h, the attention about 2 T^2 n_h (d_h+d_r)
 * against 2 T^2 n_h (2 d_c + d_r) absorbed).  K, V and the query are rounded to bf16.
 * q_nope device [n_queries, n_h, d_h]; q_rope device [n_queries, n_h, d_r] (not rotated);
 * w_uk, w_uv device [d_c, n_h*d_h]; o device [n_queries, n_h*d_h]; lse device float
 * [n_queries, n_h].  workspace: device, 256-byte aligned, at least
 * mla_prefill_unabsorbed_workspace_size() bytes (the gathered cache rows, K, V and the rotated
 * query; about 1 GB at L = T = 8192).  Needs cfg->dtype == MLA_BF16, d_nope == 128,
 * d_rope == 64, d_latent a multiple of 64, a plain cache and sm_103 (else MLA_ERR_UNSUPPORTED).
 * n_queries == 0 is a no-op. */
MLA_API mla_status mla_prefill_unabsorbed_workspace_size(const mla_config* cfg, int32_t q_start,
                                                         int32_t n_queries, size_t* bytes);
MLA_API mla_status mla_prefill_unabsorbed(const mla_config* cfg, const mla_cache* cache, int32_t seq,
                                          int32_t q_start, int32_t n_queries, const void* q_nope,
                                          const void* q_rope, const void* w_uk, const void* w_uv,
                                          void* o, float* lse, void* workspace,
                                          size_t workspace_bytes, mla_stream_t stream);

/* mla_out - absorbed output up-projection ([OPN] s.2 "V = c_kv @ W_UV", folded into the
 * output side as [GLO] describes):  o[n, h*d_h:(h+1)*d_h] = o_lat[n,h,:] @ W_UV[:, h*d_h:(h+1)*d_h]
 * o_lat device [n_tokens, n_h, d_c]; w_uv device [d_c, n_h*d_h]; o device [n_tokens, n_h*d_h].
 * n_tokens == 0 is a no-op. */
MLA_API mla_status mla_out(const mla_config* cfg, const void* o_lat, const void* w_uv, void* o,
                   int32_t n_tokens, mla_stream_t stream);

/* mla_query_proj - the query side in its simplest form ([OPN] s.2 "Q = x @ W_Q", no query
 * compression) plus the per-head RoPE query of [GLO]'s decoupled key:
 *   q_nope[n] = x[n] @ W_Q   and   q_rope[n] = x[n] @ W_QR   (q_rope unrotated: mla_absorb_q
 *   applies RoPE at the token's position)
 * x device [n_tokens, d_model]; w_q device [d_model, n_h*d_h]; w_qr device [d_model, n_h*d_r];
 * q_nope device [n_tokens, n_h, d_h]; q_rope device [n_tokens, n_h, d_r].  Rows must be
 * multiples of 16 bytes (else MLA_ERR_UNSUPPORTED).  n_tokens == 0 is a no-op. */
MLA_API mla_status mla_query_proj(const mla_config* cfg, const void* x, const void* w_q, const void* w_qr,
                          void* q_nope, void* q_rope, int32_t n_tokens, mla_stream_t stream);

/* The query side with compression ([OPN] s.4: "first c_q = x @ W_DQ, then Q = c_q @ W_UQ"; the
 * query is recomputed from x and never cached).  d_cq is the width of the query latent c_q
 * (the page gives it as d_c).  The decoupled RoPE query of [GLO] comes from the same latent:
 * q_rope = c_q @ W_QR.  Two ways to the absorbed query q_cat:
 *   mla_query_latent -> mla_query_up (q_nope, q_rope) -> mla_absorb_q, or, with W_UQ folded into
 *   W_UK once (mla_fold_uq_uk, [GLO]/[RMJ] absorption by associativity),
 *   mla_query_latent -> mla_query_up (q_rope only) -> mla_absorb_q_compressed.
 * Row widths (d_cq, n_h*d_h, n_h*d_r) must be multiples of 16 bytes (else MLA_ERR_UNSUPPORTED);
 * n_tokens == 0 is a no-op. */
/* c_q[n] = x[n] @ W_DQ.  x device [n_tokens, d_model]; w_dq device [d_model, d_cq];
 * c_q device [n_tokens, d_cq]. */
MLA_API mla_status mla_query_latent(const mla_config* cfg, int32_t d_cq, const void* x, const void* w_dq,
                                    void* c_q, int32_t n_tokens, mla_stream_t stream);
/* q_nope[n] = c_q[n] @ W_UQ and q_rope[n] = c_q[n] @ W_QR (not rotated: mla_absorb_q and
 * mla_absorb_q_compressed rotate at the token's position).  c_q device [n_tokens, d_cq];
 * w_uq device [d_cq, n_h*d_h]; w_qr device [d_cq, n_h*d_r]; q_nope device [n_tokens, n_h, d_h];
 * q_rope device [n_tokens, n_h, d_r].  Either output (with its weight) may be NULL, not both. */
MLA_API mla_status mla_query_up(const mla_config* cfg, int32_t d_cq, const void* c_q, const void* w_uq,
                                const void* w_qr, void* q_nope, void* q_rope, int32_t n_tokens,
                                mla_stream_t stream);
/* W_UQ folded into W_UK, once when the weights are loaded (not a per-token step):
 *   w_uqk[:, h*d_c:(h+1)*d_c] = W_UQ[:, h*d_h:(h+1)*d_h] @ W_UK[:, h*d_h:(h+1)*d_h]^T
 * w_uq device [d_cq, n_h*d_h]; w_uk device [d_c, n_h*d_h]; w_uqk device [d_cq, n_h*d_c] (output;
 * fp32 accumulation, rounded to cfg->dtype).  For d_cq = d_c the folded weight holds n_h d_c^2
 * numbers against 2 n_h d_c d_h for the pair: twice the bytes a decode step streams at d_h =
 * d_c / 4, in exchange for one GEMM per step instead of two. */
MLA_API mla_status mla_fold_uq_uk(const mla_config* cfg, int32_t d_cq, const void* w_uq, const void* w_uk,
                                  void* w_uqk, mla_stream_t stream);
/* The absorbed query from the query latent:
 *   q_cat[n,h,0:d_c] = c_q[n] @ w_uqk[:, h*d_c:(h+1)*d_c]
 *   q_cat[n,h,d_c:W] = RoPE(q_rope[n,h,:], pos[n])
 * c_q device [n_tokens, d_cq]; q_rope device [n_tokens, n_h, d_r] (not rotated); pos device int32
 * [n_tokens]; w_uqk device [d_cq, n_h*d_c] (from mla_fold_uq_uk); q_cat device [n_tokens, n_h, W].
 * Same output as mla_absorb_q on q_nope = c_q @ W_UQ, up to rounding. */
MLA_API mla_status mla_absorb_q_compressed(const mla_config* cfg, int32_t d_cq, const void* c_q,
                                           const void* q_rope, const int32_t* pos, const void* w_uqk,
                                           void* q_cat, int32_t n_tokens, mla_stream_t stream);

/* mla_out_proj - the final projection over the concatenated heads ([OPN] s.2 "out = O @ W_O";
 * row block h of W_O belongs to head h):  out[n, :] = o[n, :] @ W_O
 * o device [n_tokens, n_h*d_h] (what mla_out writes); w_o device [n_h*d_h, d_model];
 * out device [n_tokens, d_model].  Rows of o and out must be multiples of 16 bytes
 * (else MLA_ERR_UNSUPPORTED).  n_tokens == 0 is a no-op. */
MLA_API mla_status mla_out_proj(const mla_config* cfg, const void* o, const void* w_o, void* out,
                        int32_t n_tokens, mla_stream_t stream);

/* Synchronise `stream`, then read and clear the current device's error word.
 * Returns MLA_OK, MLA_ERR_DEVICE_BOUNDS, MLA_ERR_DEVICE_TIMEOUT or MLA_ERR_CUDA. */
MLA_API mla_status mla_get_device_error(mla_stream_t stream);

/* Process-wide tuning / test knobs (not needed for normal use).  Returns the previous value. */
typedef enum {
    MLA_TUNE_ATTN_UNITS = 0,   /* >0: number of split units for decode/prefill (test use)    */
    MLA_TUNE_FORCE_SIMT = 1,   /* 1: run the portable SIMT kernels even where tcgen05 applies */
    MLA_TUNE_WAIT_LIMIT_US = 2, /* device bounded-wait limit in microseconds (default 2e6)  */
    MLA_TUNE_GEMM_HEADS = 3,   /* >0: heads per CTA of the tcgen05 projection GEMMs          */
    MLA_TUNE_GEMM_STAGES = 4,  /* >0: ring depth of the tcgen05 projection GEMMs             */
    MLA_TUNE_NO_PDL = 5,       /* 1: launch without programmatic dependent launch            */
    MLA_TUNE_SCHEDULE = 6,     /* split schedule: 0 automatic, 1 flat page partition only     */
    MLA_TUNE_GEMM_KSPLIT = 7   /* >0: K split (cluster size, <= 8) of the tcgen05 GEMMs      */
} mla_tuning_key;
MLA_API int32_t mla_set_tuning(int32_t key, int32_t value);

/* Timing hook for benchmarks: when both are non-NULL, the next mla_decode / mla_prefill /
 * mla_prefill_unabsorbed calls on this thread record `before` (a cudaEvent_t) on their stream
 * immediately before the attention kernel and `after` immediately after it, so the caller can
 * time that kernel alone.  Pass NULLs to stop.  The events stay owned by the caller. */
MLA_API void mla_set_attention_events(void* before, void* after);

/* Number of CUDA kernels this process has launched through libmla so far. */
MLA_API uint64_t mla_kernel_launches(void);

/* Which kernel family the last attention call on this thread used:
 * 0 none yet, 1 SIMT, 2 tcgen05 (absorbed), 3 tcgen05 un-absorbed causal (mla_prefill_unabsorbed). */
MLA_API int32_t mla_last_attention_path(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H */
