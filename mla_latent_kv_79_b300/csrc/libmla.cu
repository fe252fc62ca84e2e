// libmla: C ABI of the MLA latent-KV hot path (declarations and contracts in include/mla.h).
//
// One translation unit holds every kernel so the per-device error word is a single symbol.
#include <cuda_runtime.h>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "mla.h"
#include "mla_common.cuh"
#include "sched.cuh"
#include "simt_gemm.cuh"
#include "simt_attention.cuh"
#include "tc_attention.cuh"
#include "tc_gemm.cuh"
#include "tc_flash.cuh"

namespace mla {

// ----------------------------------------------------------------------------- device info
struct DeviceInfo {
    std::atomic<bool> ready{false};  // published after the fields below are filled in
    int sms = 0, smem_optin = 0, cc_major = 0, cc_minor = 0;
};
static DeviceInfo g_dev[64];
static std::mutex g_dev_mu;

static mla_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
    DeviceInfo& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
                return MLA_ERR_CUDA;
            // one shared-memory carve-out for every kernel of the library, so consecutive
            // launches of the hot path never wait for an SM to re-partition L1 and shared memory
            const void* fns[] = {
                (const void*)simt_gemm_kernel<bf16, EPI_STORE>, (const void*)simt_gemm_kernel<float, EPI_STORE>,
                (const void*)simt_gemm_kernel<bf16, EPI_APPEND>, (const void*)simt_gemm_kernel<float, EPI_APPEND>,
                (const void*)rope_query_kernel<bf16>, (const void*)rope_query_kernel<float>,
                (const void*)simt_attention_kernel<bf16, KV_PLAIN>, (const void*)simt_attention_kernel<float, KV_PLAIN>,
                (const void*)simt_attention_kernel<bf16, KV_MXFP8>, (const void*)simt_attention_kernel<float, KV_MXFP8>,
                (const void*)simt_attention_kernel<bf16, KV_MXFP4>, (const void*)simt_attention_kernel<float, KV_MXFP4>,
                (const void*)combine_kernel<bf16>, (const void*)combine_kernel<float>,
                (const void*)tca::tc_attention_kernel<KV_PLAIN>, (const void*)tca::tc_attention_kernel<KV_MXFP8>,
                (const void*)tca::tc_attention_kernel<KV_MXFP4>, (const void*)tcg::tc_gemm_kernel<tcg::ABSORB>,
                (const void*)tcg::tc_gemm_kernel<tcg::OUT>, (const void*)tcg::tc_gemm_kernel<tcg::APPEND>,
                (const void*)tcg::tc_gemm_kernel<tcg::OPROJ>, (const void*)tcg::tc_gemm_kernel<tcg::ABSORBC>,
                (const void*)tcf::prep_kernel,
                (const void*)tcf::flash_kernel};
            for (const void* f : fns)
                if (cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
                    return MLA_ERR_CUDA;
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return MLA_OK;
}

// ----------------------------------------------------------------------------- knobs
static std::atomic<int> g_tune[8] = {{0}, {0}, {2000000}, {0}, {0}, {0}, {0}, {0}};
static thread_local int g_last_path = 0;
static thread_local cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;
static std::atomic<unsigned long long> g_launches{0};

static void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static size_t elem_size(const mla_config* c) { return c->dtype == MLA_BF16 ? 2 : 4; }

static mla_status check_config(const mla_config* c) {
    if (!c) return MLA_ERR_INVALID_ARG;
    if (c->dtype != MLA_F32 && c->dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
    if (c->n_heads <= 0 || c->d_nope <= 0 || c->d_rope <= 0 || c->d_latent <= 0 ||
        c->d_model <= 0 || c->page_size <= 0)
        return MLA_ERR_INVALID_ARG;
    if ((c->d_rope & 1) || (c->d_latent & 1)) return MLA_ERR_INVALID_ARG;
    if (c->d_latent % 8) return MLA_ERR_UNSUPPORTED;  // 16-byte groups of the split partials
    if (!(c->rope_base > 0.f) || !std::isfinite(c->rope_base)) return MLA_ERR_INVALID_ARG;
    if (c->softmax_scale < 0.f || !std::isfinite(c->softmax_scale)) return MLA_ERR_INVALID_ARG;
    // row widths in bytes must keep 16-byte alignment of every row
    const size_t es = elem_size(c);
    if (((size_t)(c->d_latent + c->d_rope) * es) % 16 || ((size_t)c->d_latent * es) % 16)
        return MLA_ERR_UNSUPPORTED;
    if (c->d_latent + c->d_rope > 1024 || c->d_latent > 1024 || c->d_rope > 1024) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

static mla_status check_cache(const mla_config* c, const mla_cache* k) {
    if (!k || !k->pool || !k->page_table || k->num_pages <= 0 || k->max_pages <= 0 || k->batch <= 0)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(k->pool)) return MLA_ERR_INVALID_ARG;
    if (k->kv_format != MLA_KV_PLAIN) {
        if (k->kv_format != MLA_KV_MXFP8 && k->kv_format != MLA_KV_MXFP4) return MLA_ERR_INVALID_ARG;
        if (!k->kv_scales || !aligned16(k->kv_scales)) return MLA_ERR_INVALID_ARG;
        if ((c->d_latent + c->d_rope) % MX_BLOCK) return MLA_ERR_UNSUPPORTED;
    }
    if ((long long)k->max_pages * c->page_size > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

static float scale_of(const mla_config* c) {
    return c->softmax_scale > 0.f ? c->softmax_scale : (float)(1.0 / std::sqrt((double)(c->d_nope + c->d_rope)));
}

static mla_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

static int max_units(const DeviceInfo* d) { return d->sms > 0 ? d->sms : 148; }

static tcg::Tuning gemm_tuning(unsigned long long wait_ns) {
    tcg::Tuning t;
    t.wait_ns = wait_ns;
    t.hpc = g_tune[MLA_TUNE_GEMM_HEADS].load();
    t.stages = g_tune[MLA_TUNE_GEMM_STAGES].load();
    t.ksplit = g_tune[MLA_TUNE_GEMM_KSPLIT].load();
    t.pdl = g_tune[MLA_TUNE_NO_PDL].load() == 0;
    return t;
}

// ----------------------------------------------------------------------------- attention
template <typename T, int KVF>
static void launch_simt_attention(dim3 grid, size_t smem, cudaStream_t stream, const AttnArgs& a, int hg) {
    cudaFuncSetAttribute(simt_attention_kernel<T, KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    simt_attention_kernel<T, KVF><<<grid, 256, smem, stream>>>(a, hg);
}

static mla_status attention(const mla_config* cfg, const mla_cache* cache, QuerySet qs,
                            const void* q_cat, void* o_lat, float* lse, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
    DeviceInfo* dev;
    mla_status st = device_info(&dev);
    if (st != MLA_OK) return st;
    if (qs.n_queries == 0) return MLA_OK;
    if (!q_cat || !o_lat || !lse || !aligned16(q_cat) || !aligned16(o_lat) || !aligned16(lse))
        return MLA_ERR_INVALID_ARG;
    size_t need = 0;
    mla_workspace_size(cfg, &need);
    if (!ws || ws_bytes < need || !aligned16(ws)) return MLA_ERR_WORKSPACE;

    const int n_h = cfg->n_heads, d_c = cfg->d_latent, W = cfg->d_latent + cfg->d_rope;
    const int U_max = max_units(dev);
    AttnArgs a;
    a.qs = qs;
    a.q_cat = q_cat;
    a.pool = cache->pool;
    a.scales = cache->kv_scales;
    a.page_table = cache->page_table;
    a.max_pages = cache->max_pages;
    a.num_pages = cache->num_pages;
    a.o_lat = o_lat;
    a.lse = lse;
    a.part_o = ws;  // partials sized as fp32 (an upper bound for either dtype), then the lse slots
    a.part_lse = reinterpret_cast<float*>(ws) + (size_t)2 * U_max * n_h * d_c;
    a.n_h = n_h;
    a.d_c = d_c;
    a.width = W;
    a.scale = scale_of(cfg);
    a.qs.flat_only = g_tune[MLA_TUNE_SCHEDULE].load() == 1 ? 1 : 0;

    const int forced = g_tune[MLA_TUNE_ATTN_UNITS].load();
    const bool use_tc = !g_tune[MLA_TUNE_FORCE_SIMT].load() && tc_attention_supported(cfg, cache, dev->cc_major, dev->cc_minor);
    const bool timed = g_ev_before && g_ev_after;
    if (use_tc) {
        int U = forced > 0 ? (forced < U_max / 2 ? forced : U_max / 2) : U_max / 2;
        a.n_units = U;
        if (timed) cudaEventRecord(g_ev_before, stream);
        st = tc_attention_launch(a, cache, (unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull,
                                 g_tune[MLA_TUNE_NO_PDL].load() == 0, stream);
        if (timed) cudaEventRecord(g_ev_after, stream);
        if (st != MLA_OK) return st;
        count_launches(1);
        g_last_path = 2;
    } else {
        int hg = n_h < 16 ? n_h : 16;
        size_t smem = simt_attn_smem_bytes(hg, W, d_c);
        while (smem > (size_t)dev->smem_optin && hg > 1) { hg /= 2; smem = simt_attn_smem_bytes(hg, W, d_c); }
        if (smem > (size_t)dev->smem_optin) return MLA_ERR_UNSUPPORTED;
        int U = forced > 0 ? (forced < U_max ? forced : U_max) : U_max;
        a.n_units = U;
        dim3 grid(U, (n_h + hg - 1) / hg);
        if (timed) cudaEventRecord(g_ev_before, stream);
        if (cfg->dtype == MLA_BF16) {
            switch (cache->kv_format) {
                case MLA_KV_MXFP8: launch_simt_attention<bf16, KV_MXFP8>(grid, smem, stream, a, hg); break;
                case MLA_KV_MXFP4: launch_simt_attention<bf16, KV_MXFP4>(grid, smem, stream, a, hg); break;
                default: launch_simt_attention<bf16, KV_PLAIN>(grid, smem, stream, a, hg); break;
            }
        } else {
            switch (cache->kv_format) {
                case MLA_KV_MXFP8: launch_simt_attention<float, KV_MXFP8>(grid, smem, stream, a, hg); break;
                case MLA_KV_MXFP4: launch_simt_attention<float, KV_MXFP4>(grid, smem, stream, a, hg); break;
                default: launch_simt_attention<float, KV_PLAIN>(grid, smem, stream, a, hg); break;
            }
        }
        if (timed) cudaEventRecord(g_ev_after, stream);
        if ((st = launch_status()) != MLA_OK) return st;
        count_launches(1);
        g_last_path = 1;
    }
    // the combine is a programmatic dependent of the attention kernel: it may start early and
    // waits (griddepcontrol.wait) for the attention grid's results before reading partials
    cudaLaunchConfig_t lc = {};
    const int vec = cfg->dtype == MLA_BF16 ? 8 : 4;  // partial values per 16 bytes
    lc.gridDim = dim3(qs.n_queries, (unsigned)((n_h * (d_c / vec) + COMBINE_THREADS - 1) / COMBINE_THREADS));
    lc.blockDim = dim3(COMBINE_THREADS);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = g_tune[MLA_TUNE_NO_PDL].load() ? 0 : 1;
    cudaError_t e = cfg->dtype == MLA_BF16 ? cudaLaunchKernelEx(&lc, combine_kernel<bf16>, a)
                                           : cudaLaunchKernelEx(&lc, combine_kernel<float>, a);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    count_launches(1);
    return launch_status();
}

}  // namespace mla

using namespace mla;

extern "C" {

int32_t mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported dimensions";
        case MLA_ERR_CUDA: return "CUDA error";
        case MLA_ERR_WORKSPACE: return "workspace missing or too small";
        case MLA_ERR_DEVICE_TIMEOUT: return "device bounded wait timed out";
        case MLA_ERR_DEVICE_BOUNDS: return "page id or position outside the cache";
        case MLA_ERR_SCRATCH_LIMIT: return "configuration needs more split scratch than the fixed no-allocation array holds";
    }
    return "unknown status";
}

int32_t mla_set_tuning(int32_t key, int32_t value) {
    if (key < 0 || key > 7) return -1;
    if (key == MLA_TUNE_WAIT_LIMIT_US && value <= 0) value = 2000000;
    return g_tune[key].exchange(value);
}

int32_t mla_last_attention_path(void) { return g_last_path; }

void mla_set_attention_events(void* before, void* after) {
    g_ev_before = reinterpret_cast<cudaEvent_t>(before);
    g_ev_after = reinterpret_cast<cudaEvent_t>(after);
}

uint64_t mla_kernel_launches(void) { return g_launches.load(); }

mla_status mla_workspace_size(const mla_config* cfg, size_t* bytes) {
    if (!bytes) return MLA_ERR_INVALID_ARG;
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    const size_t slots = 2 * (size_t)max_units(dev);
    size_t b = slots * (size_t)cfg->n_heads * ((size_t)cfg->d_latent + 1) * sizeof(float);
    *bytes = (b + 255) & ~(size_t)255;
    return MLA_OK;
}

mla_status mla_cache_append(const mla_config* cfg, const mla_cache* cache, const void* x,
                            const void* w_dkv, const void* w_kr, const int32_t* seq_idx,
                            const int32_t* pos, int32_t n_tokens, mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if ((st = check_cache(cfg, cache)) != MLA_OK) return st;
    if (n_tokens < 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!x || !w_dkv || !w_kr || !seq_idx || !pos) return MLA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_dkv) || !aligned16(w_kr)) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int W = cfg->d_latent + cfg->d_rope;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    const bool tc_ok = tc_gemm_append_supported(cfg, n_tokens, dev->cc_major, dev->cc_minor) &&
                       (long long)cache->num_pages * cfg->page_size < (1LL << 31);
    if (cache->kv_format != MLA_KV_PLAIN && !tc_ok) return MLA_ERR_UNSUPPORTED;  // MX encoding: tensor-core path only
    if ((!g_tune[MLA_TUNE_FORCE_SIMT].load() || cache->kv_format != MLA_KV_PLAIN) && tc_ok) {
        st = tc_gemm_append(cfg, cache, x, w_dkv, w_kr, seq_idx, pos, n_tokens,
                            gemm_tuning((unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull), s);
        if (st == MLA_OK) count_launches(1);
        return st;
    }
    SimtGemmArgs g{};
    g.A = x; g.lda = cfg->d_model; g.a_batch = 0;
    g.B = w_dkv; g.ldb_k = cfg->d_latent; g.ldb_n = 1; g.b_batch = 0;
    g.B2 = w_kr; g.ldb2_k = cfg->d_rope; g.n_split = cfg->d_latent;
    g.C = cache->pool;
    g.M = n_tokens; g.N = W; g.K = cfg->d_model;
    g.seq_idx = seq_idx; g.pos = pos;
    g.page_table = cache->page_table; g.max_pages = cache->max_pages; g.batch = cache->batch;
    g.page_size = cfg->page_size; g.num_pages = cache->num_pages; g.width = W;
    rope_freq_fill(&g.rf, cfg->d_rope, cfg->rope_base);
    dim3 grid((W + 63) / 64, (n_tokens + 63) / 64, 1);
    if (cfg->dtype == MLA_BF16) simt_gemm_kernel<bf16, EPI_APPEND><<<grid, 256, 0, s>>>(g);
    else simt_gemm_kernel<float, EPI_APPEND><<<grid, 256, 0, s>>>(g);
    count_launches(1);
    return launch_status();
}

mla_status mla_absorb_q(const mla_config* cfg, const void* q_nope, const void* q_rope,
                        const int32_t* pos, const void* w_uk, void* q_cat, int32_t n_tokens,
                        mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (n_tokens < 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!q_nope || !q_rope || !pos || !w_uk || !q_cat) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_cat))
        return MLA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int n_h = cfg->n_heads, d_h = cfg->d_nope, d_c = cfg->d_latent, d_r = cfg->d_rope;
    const int W = d_c + d_r;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    const unsigned long long wait_ns = (unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull;
    if (!g_tune[MLA_TUNE_FORCE_SIMT].load() && tc_gemm_absorb_supported(cfg, n_tokens, dev->cc_major, dev->cc_minor)) {
        // one tcgen05 kernel writes both halves of q_cat
        st = tc_gemm_absorb(cfg, q_nope, q_rope, pos, w_uk, q_cat, n_tokens, gemm_tuning(wait_ns), s);
        if (st != MLA_OK) return st;
        count_launches(1);
        return MLA_OK;
    }
    const dim3 blocks(n_tokens, (n_h + ROPE_HEADS - 1) / ROPE_HEADS);
    RopeFreq rf;
    rope_freq_fill(&rf, d_r, cfg->rope_base);
    if (cfg->dtype == MLA_BF16)
        rope_query_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)q_rope, pos, (bf16*)q_cat, n_tokens, n_h, d_r, d_c, rf);
    else
        rope_query_kernel<float><<<blocks, 256, 0, s>>>((const float*)q_rope, pos, (float*)q_cat, n_tokens, n_h, d_r, d_c, rf);
    count_launches(1);
    if ((st = launch_status()) != MLA_OK) return st;
    SimtGemmArgs g{};
    g.A = q_nope; g.lda = (long long)n_h * d_h; g.a_batch = d_h;
    g.B = w_uk; g.ldb_k = 1; g.ldb_n = (long long)n_h * d_h; g.b_batch = d_h;  // B(j,c) = W_UK[c, h*d_h+j]
    g.C = q_cat; g.ldc = (long long)n_h * W; g.c_batch = W;
    g.M = n_tokens; g.N = d_c; g.K = d_h;
    dim3 grid((d_c + 63) / 64, (n_tokens + 63) / 64, n_h);
    if (cfg->dtype == MLA_BF16) simt_gemm_kernel<bf16, EPI_STORE><<<grid, 256, 0, s>>>(g);
    else simt_gemm_kernel<float, EPI_STORE><<<grid, 256, 0, s>>>(g);
    count_launches(1);
    if ((st = launch_status()) != MLA_OK) return st;
    return MLA_OK;
}

mla_status mla_decode(const mla_config* cfg, const mla_cache* cache, const void* q_cat,
                      void* o_lat, float* lse, void* workspace, size_t workspace_bytes,
                      mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if ((st = check_cache(cfg, cache)) != MLA_OK) return st;
    if (!cache->seq_lens) return MLA_ERR_INVALID_ARG;
    QuerySet qs{};
    qs.mode = 0;
    qs.n_queries = cache->batch;
    qs.seq_lens = cache->seq_lens;
    qs.page_size = cfg->page_size;
    qs.max_len = cache->max_pages * cfg->page_size;
    return attention(cfg, cache, qs, q_cat, o_lat, lse, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ----------------------------------------------------------------------------- no-allocation decode
// mla_decode_static is for callers that cannot allocate per call or hand in a buffer: a plain C
// host program without a device allocator, or a serving loop in which cudaMalloc / cudaFree
// (which may synchronise the device) are not allowed between steps.  Its split partials live
// in this file-scope array, one per device, created with the module: the call allocates
// nothing.  Nothing in it has to start at zero (each partial the combine reads is written
// earlier in the same call); calls that overlap in time race on it.
namespace mla {
static __device__ __align__(256) unsigned char g_static_scratch[MLA_STATIC_SCRATCH_BYTES];
static void* g_static_ptr[64];
static std::mutex g_static_mu;

// Device address of g_static_scratch on the current device, looked up once per device (with
// that device current) by the first call.
static mla_status static_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress((void**)&ptr, g_static_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return MLA_ERR_CUDA;
        }
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return MLA_OK;
}
}  // namespace mla

extern "C" {

mla_status mla_decode_static(const mla_config* cfg, const mla_cache* cache, const void* q_cat,
                             void* o_lat, float* lse, mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    size_t need = 0;
    if ((st = mla_workspace_size(cfg, &need)) != MLA_OK) return st;
    if (need > MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if ((st = static_scratch(&scratch)) != MLA_OK) return st;
    return mla_decode(cfg, cache, q_cat, o_lat, lse, scratch, MLA_STATIC_SCRATCH_BYTES, stream);
}

mla_status mla_prefill(const mla_config* cfg, const mla_cache* cache, int32_t seq,
                       int32_t q_start, int32_t n_queries, const void* q_cat, void* o_lat,
                       float* lse, void* workspace, size_t workspace_bytes, mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if ((st = check_cache(cfg, cache)) != MLA_OK) return st;
    if (seq < 0 || seq >= cache->batch || q_start < 0 || n_queries < 0) return MLA_ERR_INVALID_ARG;
    if ((long long)q_start + n_queries > (long long)cache->max_pages * cfg->page_size)
        return MLA_ERR_INVALID_ARG;
    QuerySet qs{};
    qs.mode = 1;
    qs.n_queries = n_queries;
    qs.seq = seq;
    qs.q_start = q_start;
    qs.page_size = cfg->page_size;
    qs.max_len = cache->max_pages * cfg->page_size;
    return attention(cfg, cache, qs, q_cat, o_lat, lse, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

static bool unabsorbed_supported(const mla_config* c, const mla_cache* k, const DeviceInfo* d) {
    return c->dtype == MLA_BF16 && c->d_nope == tcf::DH && c->d_rope == tcf::DR && c->d_latent % 64 == 0 &&
           d->cc_major == 10 && d->cc_minor == 3 && k->kv_format == MLA_KV_PLAIN;
}

mla_status mla_prefill_unabsorbed_workspace_size(const mla_config* cfg, int32_t q_start, int32_t n_queries,
                                                  size_t* bytes) {
    if (!bytes || q_start < 0 || n_queries < 0) return MLA_ERR_INVALID_ARG;
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    *bytes = tcf::unabsorbed_ws(cfg->n_heads, cfg->d_nope, cfg->d_rope, cfg->d_latent + cfg->d_rope,
                                (long long)q_start + n_queries, n_queries).total;
    return MLA_OK;
}

mla_status mla_prefill_unabsorbed(const mla_config* cfg, const mla_cache* cache, int32_t seq, int32_t q_start,
                                  int32_t n_queries, const void* q_nope, const void* q_rope, const void* w_uk,
                                  const void* w_uv, void* o, float* lse, void* workspace, size_t workspace_bytes,
                                  mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if ((st = check_cache(cfg, cache)) != MLA_OK) return st;
    if (seq < 0 || seq >= cache->batch || q_start < 0 || n_queries < 0) return MLA_ERR_INVALID_ARG;
    if ((long long)q_start + n_queries > (long long)cache->max_pages * cfg->page_size) return MLA_ERR_INVALID_ARG;
    if (n_queries == 0) return MLA_OK;
    if (!q_nope || !q_rope || !w_uk || !w_uv || !o || !lse) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(o) ||
        !aligned16(lse))
        return MLA_ERR_INVALID_ARG;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    if (!unabsorbed_supported(cfg, cache, dev) || (long long)cfg->n_heads * n_queries >= (1LL << 31))
        return MLA_ERR_UNSUPPORTED;
    const int W = cfg->d_latent + cfg->d_rope, n_h = cfg->n_heads;
    const long long L = (long long)q_start + n_queries;
    const tcf::UnabsorbedWs ws = tcf::unabsorbed_ws(n_h, cfg->d_nope, cfg->d_rope, W, L, n_queries);
    if (!workspace || workspace_bytes < ws.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MLA_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* w8 = reinterpret_cast<uint8_t*>(workspace);
    bf16* rows = reinterpret_cast<bf16*>(w8 + ws.rows);
    bf16* K = reinterpret_cast<bf16*>(w8 + ws.k);
    bf16* V = reinterpret_cast<bf16*>(w8 + ws.v);
    bf16* qu = reinterpret_cast<bf16*>(w8 + ws.qu);
    const bool pdl = g_tune[MLA_TUNE_NO_PDL].load() == 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    // 1. gather the sequence's rows and build the un-absorbed query
    tcf::PrepArgs p{};
    p.pool = reinterpret_cast<const bf16*>(cache->pool);
    p.page_row = cache->page_table + (size_t)seq * cache->max_pages;
    p.max_pages = cache->max_pages;
    p.num_pages = cache->num_pages;
    p.page_size = cfg->page_size;
    p.width = W;
    p.n_keys = (int)L;
    p.rows = rows;
    p.q_nope = reinterpret_cast<const bf16*>(q_nope);
    p.q_rope = reinterpret_cast<const bf16*>(q_rope);
    p.n_queries = n_queries;
    p.n_h = n_h;
    p.q_start = q_start;
    rope_freq_fill(&p.rf, cfg->d_rope, cfg->rope_base);
    p.qu = qu;
    const long long groups = L * (W / 8) + (long long)n_queries * n_h * ((tcf::DH + tcf::DR) / 8);
    long long blocks = (groups + 255) / 256;
    if (blocks > 8LL * max_units(dev)) blocks = 8LL * max_units(dev);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)blocks);
    lc.blockDim = dim3(256);
    lc.stream = s;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&lc, tcf::prep_kernel, p) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    count_launches(1);
    // 2. K = c_kv . W_UK and V = c_kv . W_UV over the gathered rows (row pitch W)
    const tcg::Tuning tu = gemm_tuning((unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull);
    const long long hd = (long long)n_h * cfg->d_nope;
    if ((st = tc_gemm_dense(cfg, rows, w_uk, K, cfg->d_latent, hd, (int)L, tu, s, W)) != MLA_OK) return st;
    count_launches(1);
    if ((st = tc_gemm_dense(cfg, rows, w_uv, V, cfg->d_latent, hd, (int)L, tu, s, W)) != MLA_OK) return st;
    count_launches(1);
    // 3. causal attention per (head, 128-query tile)
    CUtensorMap tmq, tmk, tmr, tmv;
    if (!tcf::encode_map(&tmq, qu, tcf::DQ, (uint64_t)n_h * n_queries, tcf::DQ) ||
        !tcf::encode_map(&tmk, K, (uint64_t)hd, (uint64_t)L, (uint64_t)hd) ||
        !tcf::encode_map(&tmr, rows, (uint64_t)W, (uint64_t)L, (uint64_t)W) ||
        !tcf::encode_map(&tmv, V, (uint64_t)hd, (uint64_t)L, (uint64_t)hd))
        return MLA_ERR_CUDA;
    tcf::FlashArgs fa{};
    fa.n_queries = n_queries;
    fa.n_keys = (int)L;
    fa.n_h = n_h;
    fa.q_start = q_start;
    fa.rope_col = cfg->d_latent;
    fa.scale_log2 = scale_of(cfg) * 1.4426950408889634f;
    fa.o = reinterpret_cast<bf16*>(o);
    fa.lse = lse;
    fa.wait_ns = (unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull;
    if (cudaFuncSetAttribute(tcf::flash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tcf::SMEM_BYTES) !=
        cudaSuccess)
        return MLA_ERR_CUDA;
    const int n_qt = (n_queries + tcf::BQ - 1) / tcf::BQ;
    cudaLaunchConfig_t lf = {};
    lf.gridDim = dim3((unsigned)(n_qt * n_h));
    lf.blockDim = dim3(tcf::NTHREADS);
    lf.dynamicSmemBytes = tcf::SMEM_BYTES;
    lf.stream = s;
    lf.attrs = attr;
    lf.numAttrs = pdl ? 1 : 0;
    const bool timed = g_ev_before && g_ev_after;
    if (timed) cudaEventRecord(g_ev_before, s);
    if (cudaLaunchKernelEx(&lf, tcf::flash_kernel, tmq, tmk, tmr, tmv, fa) != cudaSuccess) {
        cudaGetLastError();
        return MLA_ERR_CUDA;
    }
    if (timed) cudaEventRecord(g_ev_after, s);
    count_launches(1);
    g_last_path = 3;
    return launch_status();
}

mla_status mla_out(const mla_config* cfg, const void* o_lat, const void* w_uv, void* o,
                   int32_t n_tokens, mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (n_tokens < 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!o_lat || !w_uv || !o || !aligned16(o_lat) || !aligned16(w_uv) || !aligned16(o))
        return MLA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int n_h = cfg->n_heads, d_h = cfg->d_nope, d_c = cfg->d_latent;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    if (!g_tune[MLA_TUNE_FORCE_SIMT].load() && tc_gemm_out_supported(cfg, n_tokens, dev->cc_major, dev->cc_minor)) {
        st = tc_gemm_out(cfg, o_lat, w_uv, o, n_tokens,
                         gemm_tuning((unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull), s);
        if (st == MLA_OK) count_launches(1);
        return st;
    }
    SimtGemmArgs g{};
    g.A = o_lat; g.lda = (long long)n_h * d_c; g.a_batch = d_c;
    g.B = w_uv; g.ldb_k = (long long)n_h * d_h; g.ldb_n = 1; g.b_batch = d_h;   // B(c,j) = W_UV[c, h*d_h+j]
    g.C = o; g.ldc = (long long)n_h * d_h; g.c_batch = d_h;
    g.M = n_tokens; g.N = d_h; g.K = d_c;
    dim3 grid((d_h + 63) / 64, (n_tokens + 63) / 64, n_h);
    if (cfg->dtype == MLA_BF16) simt_gemm_kernel<bf16, EPI_STORE><<<grid, 256, 0, s>>>(g);
    else simt_gemm_kernel<float, EPI_STORE><<<grid, 256, 0, s>>>(g);
    count_launches(1);
    return launch_status();
}

static mla_status dense_projection(const mla_config* cfg, const DeviceInfo* dev, const void* in, const void* w,
                                   void* out, long long K, long long M, int32_t n_tokens, cudaStream_t s);

mla_status mla_out_proj(const mla_config* cfg, const void* o, const void* w_o, void* out, int32_t n_tokens,
                        mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (n_tokens < 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!o || !w_o || !out || !aligned16(o) || !aligned16(w_o) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
    const long long hd = (long long)cfg->n_heads * cfg->d_nope;
    const int dm = cfg->d_model;
    const size_t es = elem_size(cfg);
    if (((size_t)hd * es) % 16 || ((size_t)dm * es) % 16 || hd > (1LL << 30)) return MLA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    return dense_projection(cfg, dev, o, w_o, out, hd, dm, n_tokens, s);
}

// out[n, :] = in[n, :] . W (W [K, M] row-major) on the tensor cores where they apply, else the
// portable SIMT GEMM
static mla_status dense_projection(const mla_config* cfg, const DeviceInfo* dev, const void* in, const void* w,
                                   void* out, long long K, long long M, int32_t n_tokens, cudaStream_t s) {
    if (!g_tune[MLA_TUNE_FORCE_SIMT].load() && tc_gemm_dense_supported(cfg, K, M, n_tokens, dev->cc_major, dev->cc_minor)) {
        const mla_status st = tc_gemm_dense(cfg, in, w, out, K, M, n_tokens,
                                            gemm_tuning((unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull), s);
        if (st == MLA_OK) count_launches(1);
        return st;
    }
    SimtGemmArgs g{};
    g.A = in; g.lda = K; g.a_batch = 0;
    g.B = w; g.ldb_k = M; g.ldb_n = 1; g.b_batch = 0;  // B(k, m) = W[k, m]
    g.C = out; g.ldc = M; g.c_batch = 0;
    g.M = n_tokens; g.N = (int)M; g.K = (int)K;
    dim3 grid((unsigned)((M + 63) / 64), (unsigned)((n_tokens + 63) / 64), 1);
    if (cfg->dtype == MLA_BF16) simt_gemm_kernel<bf16, EPI_STORE><<<grid, 256, 0, s>>>(g);
    else simt_gemm_kernel<float, EPI_STORE><<<grid, 256, 0, s>>>(g);
    count_launches(1);
    return launch_status();
}

mla_status mla_query_proj(const mla_config* cfg, const void* x, const void* w_q, const void* w_qr, void* q_nope,
                          void* q_rope, int32_t n_tokens, mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (n_tokens < 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!x || !w_q || !w_qr || !q_nope || !q_rope || !aligned16(x) || !aligned16(w_q) || !aligned16(w_qr) ||
        !aligned16(q_nope) || !aligned16(q_rope))
        return MLA_ERR_INVALID_ARG;
    const long long hd = (long long)cfg->n_heads * cfg->d_nope, hr = (long long)cfg->n_heads * cfg->d_rope;
    const int dm = cfg->d_model;
    const size_t es = elem_size(cfg);
    if (((size_t)hd * es) % 16 || ((size_t)hr * es) % 16 || ((size_t)dm * es) % 16 || hd > (1LL << 30) ||
        hr > (1LL << 30))
        return MLA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    if ((st = dense_projection(cfg, dev, x, w_q, q_nope, dm, hd, n_tokens, s)) != MLA_OK) return st;
    return dense_projection(cfg, dev, x, w_qr, q_rope, dm, hr, n_tokens, s);
}

mla_status mla_query_latent(const mla_config* cfg, int32_t d_cq, const void* x, const void* w_dq, void* c_q,
                            int32_t n_tokens, mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (n_tokens < 0 || d_cq <= 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!x || !w_dq || !c_q || !aligned16(x) || !aligned16(w_dq) || !aligned16(c_q)) return MLA_ERR_INVALID_ARG;
    const size_t es = elem_size(cfg);
    if (((size_t)d_cq * es) % 16 || ((size_t)cfg->d_model * es) % 16) return MLA_ERR_UNSUPPORTED;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    return dense_projection(cfg, dev, x, w_dq, c_q, cfg->d_model, d_cq, n_tokens, reinterpret_cast<cudaStream_t>(stream));
}

mla_status mla_query_up(const mla_config* cfg, int32_t d_cq, const void* c_q, const void* w_uq, const void* w_qr,
                        void* q_nope, void* q_rope, int32_t n_tokens, mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (n_tokens < 0 || d_cq <= 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!c_q || !aligned16(c_q) || (!q_nope && !q_rope)) return MLA_ERR_INVALID_ARG;
    if (q_nope && (!w_uq || !aligned16(w_uq) || !aligned16(q_nope))) return MLA_ERR_INVALID_ARG;
    if (q_rope && (!w_qr || !aligned16(w_qr) || !aligned16(q_rope))) return MLA_ERR_INVALID_ARG;
    const long long hd = (long long)cfg->n_heads * cfg->d_nope, hr = (long long)cfg->n_heads * cfg->d_rope;
    const size_t es = elem_size(cfg);
    if (((size_t)d_cq * es) % 16 || ((size_t)hd * es) % 16 || ((size_t)hr * es) % 16) return MLA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    if (q_nope && (st = dense_projection(cfg, dev, c_q, w_uq, q_nope, d_cq, hd, n_tokens, s)) != MLA_OK) return st;
    if (q_rope && (st = dense_projection(cfg, dev, c_q, w_qr, q_rope, d_cq, hr, n_tokens, s)) != MLA_OK) return st;
    return MLA_OK;
}

mla_status mla_fold_uq_uk(const mla_config* cfg, int32_t d_cq, const void* w_uq, const void* w_uk, void* w_uqk,
                          mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (d_cq <= 0 || !w_uq || !w_uk || !w_uqk) return MLA_ERR_INVALID_ARG;
    if (!aligned16(w_uq) || !aligned16(w_uk) || !aligned16(w_uqk)) return MLA_ERR_INVALID_ARG;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int n_h = cfg->n_heads, d_h = cfg->d_nope, d_c = cfg->d_latent;
    // per head h: W_UQK[k, h*d_c + c] = sum_j W_UQ[k, h*d_h + j] * W_UK[c, h*d_h + j]  (a weight-load
    // step, once; fp32 accumulation)
    SimtGemmArgs g{};
    g.A = w_uq; g.lda = (long long)n_h * d_h; g.a_batch = d_h;
    g.B = w_uk; g.ldb_k = 1; g.ldb_n = (long long)n_h * d_h; g.b_batch = d_h;  // B(j, c) = W_UK[c, h*d_h + j]
    g.C = w_uqk; g.ldc = (long long)n_h * d_c; g.c_batch = d_c;
    g.M = d_cq; g.N = d_c; g.K = d_h;
    dim3 grid((d_c + 63) / 64, (d_cq + 63) / 64, n_h);
    if (cfg->dtype == MLA_BF16) simt_gemm_kernel<bf16, EPI_STORE><<<grid, 256, 0, s>>>(g);
    else simt_gemm_kernel<float, EPI_STORE><<<grid, 256, 0, s>>>(g);
    count_launches(1);
    return launch_status();
}

mla_status mla_absorb_q_compressed(const mla_config* cfg, int32_t d_cq, const void* c_q, const void* q_rope,
                                   const int32_t* pos, const void* w_uqk, void* q_cat, int32_t n_tokens,
                                   mla_stream_t stream) {
    mla_status st = check_config(cfg);
    if (st != MLA_OK) return st;
    if (n_tokens < 0 || d_cq <= 0) return MLA_ERR_INVALID_ARG;
    if (n_tokens == 0) return MLA_OK;
    if (!c_q || !q_rope || !pos || !w_uqk || !q_cat) return MLA_ERR_INVALID_ARG;
    if (!aligned16(c_q) || !aligned16(q_rope) || !aligned16(w_uqk) || !aligned16(q_cat)) return MLA_ERR_INVALID_ARG;
    const size_t es = elem_size(cfg);
    if (((size_t)d_cq * es) % 16) return MLA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int n_h = cfg->n_heads, d_c = cfg->d_latent, d_r = cfg->d_rope;
    const int W = d_c + d_r;
    DeviceInfo* dev;
    if ((st = device_info(&dev)) != MLA_OK) return st;
    const unsigned long long wait_ns = (unsigned long long)g_tune[MLA_TUNE_WAIT_LIMIT_US].load() * 1000ull;
    if (!g_tune[MLA_TUNE_FORCE_SIMT].load() &&
        tc_gemm_absorbc_supported(cfg, d_cq, n_tokens, dev->cc_major, dev->cc_minor)) {
        st = tc_gemm_absorb_compressed(cfg, d_cq, c_q, q_rope, pos, w_uqk, q_cat, n_tokens, gemm_tuning(wait_ns), s);
        if (st != MLA_OK) return st;
        count_launches(1);
        return MLA_OK;
    }
    const dim3 blocks(n_tokens, (n_h + ROPE_HEADS - 1) / ROPE_HEADS);
    RopeFreq rf;
    rope_freq_fill(&rf, d_r, cfg->rope_base);
    if (cfg->dtype == MLA_BF16)
        rope_query_kernel<bf16><<<blocks, 256, 0, s>>>((const bf16*)q_rope, pos, (bf16*)q_cat, n_tokens, n_h, d_r, d_c, rf);
    else
        rope_query_kernel<float><<<blocks, 256, 0, s>>>((const float*)q_rope, pos, (float*)q_cat, n_tokens, n_h, d_r, d_c, rf);
    count_launches(1);
    if ((st = launch_status()) != MLA_OK) return st;
    SimtGemmArgs g{};
    g.A = c_q; g.lda = d_cq; g.a_batch = 0;                                              // every head reads c_q
    g.B = w_uqk; g.ldb_k = (long long)n_h * d_c; g.ldb_n = 1; g.b_batch = d_c;          // B(k, c) = W_UQK[k, h*d_c + c]
    g.C = q_cat; g.ldc = (long long)n_h * W; g.c_batch = W;
    g.M = n_tokens; g.N = d_c; g.K = d_cq;
    dim3 grid((d_c + 63) / 64, (n_tokens + 63) / 64, n_h);
    if (cfg->dtype == MLA_BF16) simt_gemm_kernel<bf16, EPI_STORE><<<grid, 256, 0, s>>>(g);
    else simt_gemm_kernel<float, EPI_STORE><<<grid, 256, 0, s>>>(g);
    count_launches(1);
    return launch_status();
}

mla_status mla_get_device_error(mla_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
    return (mla_status)v;
}

}  // extern "C"
