// Host side of the C ABI declared in include/kvq.h: argument validation,
// cache geometry, split selection, workspace carving and kernel dispatch.
// No function here allocates memory or synchronizes a stream.
#include <cuda.h>  // driver types for the context identifier (no libcuda link)
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "kvq_internal.cuh"

namespace kvq {

unsigned long long current_context_id() {
  // cuCtxGetCurrent and cuCtxGetId, looked up once through the runtime
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id + 1;  // 0 stays "unknown"
}

namespace {

constexpr size_t kAlign = 16;

bool aligned(const void* p) { return ((uintptr_t)p % kAlign) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Validates a cache descriptor; fills `g` on success.
kvq_status check_desc(const kvq_cache_desc* d, CacheGeom* g) {
  if (!d) return KVQ_ERR_INVALID_ARG;
  if (d->bits != 2 && d->bits != 4 && d->bits != 8 && d->bits != 16) return KVQ_ERR_INVALID_ARG;
  if (d->head_dim <= 0 || d->head_dim % 8 || d->num_kv_heads <= 0) return KVQ_ERR_INVALID_ARG;
  if (d->bits != 16) {
    if (d->group_size < 8 || d->group_size % 8 || d->head_dim % d->group_size)
      return KVQ_ERR_INVALID_ARG;
  }
  if (d->symmetric != 0 && d->symmetric != 1) return KVQ_ERR_INVALID_ARG;
  if (d->symmetric && d->bits == 16) return KVQ_ERR_INVALID_ARG;
  if (d->k_per_channel != 0 && d->k_per_channel != 1) return KVQ_ERR_INVALID_ARG;
  if (d->nf4 != 0 && d->nf4 != 1) return KVQ_ERR_INVALID_ARG;
  if (d->nf4 && (d->bits != 4 || d->symmetric || d->k_per_channel)) return KVQ_ERR_INVALID_ARG;
  if (d->k_per_channel) {
    if (d->bits == 16 || d->bits == 2 || d->symmetric || d->sink_tokens < 0)
      return KVQ_ERR_INVALID_ARG;
    if (d->layout == KVQ_DENSE &&
        (d->capacity % d->group_size || d->sink_tokens >= d->capacity))
      return KVQ_ERR_INVALID_ARG;
    // paged: pages of the quantized region hold whole blocks
    if (d->layout == KVQ_PAGED && d->capacity % d->group_size) return KVQ_ERR_INVALID_ARG;
  } else if (d->sink_tokens != 0) {
    return KVQ_ERR_INVALID_ARG;
  }
  if (d->layout == KVQ_DENSE) {
    if (d->capacity <= 0) return KVQ_ERR_INVALID_ARG;
  } else if (d->layout == KVQ_PAGED) {
    if (d->capacity <= 0 || d->capacity % 8 || d->num_pages <= 0 || d->max_blocks_per_seq <= 0)
      return KVQ_ERR_INVALID_ARG;
    if ((int64_t)d->capacity * d->max_blocks_per_seq + (d->k_per_channel ? d->sink_tokens : 0) >
        INT32_MAX)
      return KVQ_ERR_INVALID_ARG;
  } else {
    return KVQ_ERR_INVALID_ARG;
  }
  if (g) {
    g->bits = d->bits;
    g->D = d->head_dim;
    g->g = (d->bits == 16) ? d->head_dim : d->group_size;
    g->ngroups = (d->bits == 16) ? 0 : d->head_dim / d->group_size;
    g->row_bytes = d->head_dim * d->bits / 8;
    g->Hkv = d->num_kv_heads;
    g->layout = d->layout;
    g->slots = d->capacity;
    g->num_pages = d->layout == KVQ_PAGED ? d->num_pages : 0;
    g->max_blocks = d->layout == KVQ_PAGED ? d->max_blocks_per_seq : 0;
    g->sym = d->symmetric;
    g->kch = d->k_per_channel;
    g->sink = d->k_per_channel ? d->sink_tokens : 0;
    g->nf4 = d->nf4;
    g->block_table = nullptr;
  }
  // the kernels are built for these head sizes; byte accounting takes any
  if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

kvq_status check_cache(const kvq_cache_desc* d, const kvq_cache* c) {
  if (!c || !c->k_codes || !c->v_codes) return KVQ_ERR_INVALID_ARG;
  if (!aligned(c->k_codes) || !aligned(c->v_codes)) return KVQ_ERR_INVALID_ARG;
  if (d->bits != 16) {
    if (!c->k_scale || !c->v_scale || !aligned(c->k_scale) || !aligned(c->v_scale))
      return KVQ_ERR_INVALID_ARG;
    if (!d->symmetric && !d->nf4 &&
        (!c->k_zero || !c->v_zero || !aligned(c->k_zero) || !aligned(c->v_zero)))
      return KVQ_ERR_INVALID_ARG;
  }
  if (d->layout == KVQ_PAGED && (!c->block_table || !aligned(c->block_table)))
    return KVQ_ERR_INVALID_ARG;
  if (d->k_per_channel &&
      (!c->k_window || !c->v_window || !aligned(c->k_window) || !aligned(c->v_window)))
    return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

// A failed CUDA call maps to KVQ_ERR_CUDA; with KVQ_VERBOSE set in the
// environment its name also goes to stderr.
kvq_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return KVQ_OK;
  static const bool verbose = getenv("KVQ_VERBOSE") != nullptr;
  if (verbose) fprintf(stderr, "kvq: CUDA error %d (%s)\n", (int)e, cudaGetErrorName(e));
  return KVQ_ERR_CUDA;
}

int sm_count() {
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

int32_t split_chunk(int64_t max_len, int32_t splits) {
  return (int32_t)(ceil_div(ceil_div(std::max<int64_t>(max_len, 1), splits), kChunkAlign) * kChunkAlign);
}

// Fixed cost of one CTA (prologue, pipeline fill, partial write and merge)
// expressed in tokens of streaming work; used to weigh more splits against
// fewer (fitted to split sweeps of the tensor-core kernel on GB300).
constexpr int64_t kCtaOverheadTokens = 1024;

// Split count.  Explicit requests are honoured up to one chunk-aligned tile
// per split and need no device.  The automatic choice models the launch as
// waves of equal CTAs over (SMs x CTAs per SM) slots and minimises
// waves x (tokens per CTA + fixed CTA cost), with at least 256 tokens per split.
int32_t choose_splits(int64_t units, int64_t max_len, int32_t requested, int ctas_per_sm) {
  const int64_t L = std::max<int64_t>(max_len, 1);
  const int64_t max_splits = ceil_div(L, kChunkAlign);
  int64_t s;
  if (requested > 0) {
    s = std::min<int64_t>(requested, max_splits);
  } else {
    const int sms = sm_count();
    if (sms <= 0 || ctas_per_sm <= 0) return 0;
    const int64_t slots = (int64_t)sms * ctas_per_sm;
    const int64_t s_cap = std::max<int64_t>(1, std::min<int64_t>(ceil_div(L, 256), 256));
    int64_t best = 1;
    double best_cost = 1e300;
    for (int64_t c = 1; c <= s_cap; ++c) {
      const int64_t chunk = split_chunk(L, (int32_t)c);
      const int64_t eff = ceil_div(L, chunk);
      const int64_t waves = ceil_div(std::max<int64_t>(units, 1) * eff, slots);
      const double cost = (double)waves * (double)(chunk + kCtaOverheadTokens);
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best = eff;
      }
    }
    s = best;
  }
  s = std::max<int64_t>(1, s);
  // splits cover chunk-aligned ranges; drop splits that would be empty
  return (int32_t)ceil_div(L, split_chunk(L, (int32_t)s));
}

// NF4 levels: the (i + 1/2)/16 quantiles of N(0, 1) divided by the outermost
// one, rounded to fp16 ("Gör inference billig", NF4: the sixteen levels sit
// at the quantiles of a normal distribution).  Each quantile solves
// Phi(x) = p, Phi(x) = erfc(-x / sqrt 2) / 2, by bisection to double
// precision.  Computed once.
struct Nf4Table {
  float level[16];
  float mid[16];
  bool symmetric;  // level[15 - i] == -level[i]: the tensor-core kernel's sign-magnitude lookup
};

const Nf4Table& nf4_table() {
  static const Nf4Table t = [] {
    Nf4Table r{};
    double z[16];
    for (int i = 0; i < 16; ++i) {
      const double p = (i + 0.5) / 16.0;
      double lo = -10.0, hi = 10.0;
      for (int it = 0; it < 200; ++it) {
        const double m = 0.5 * (lo + hi);
        if (0.5 * erfc(-m / sqrt(2.0)) < p) lo = m; else hi = m;
      }
      z[i] = 0.5 * (lo + hi);
    }
    for (int i = 0; i < 16; ++i) r.level[i] = __half2float(__double2half(z[i] / z[15]));
    for (int i = 0; i < 15; ++i) r.mid[i] = (r.level[i] + r.level[i + 1]) * 0.5f;
    r.mid[15] = INFINITY;
    r.symmetric = true;
    for (int i = 0; i < 8; ++i) r.symmetric = r.symmetric && r.level[15 - i] == -r.level[i];
    return r;
  }();
  return t;
}

// Formats and shapes that may have a tensor-core kernel: INT2 / INT4 / INT8
// codes (NF4 as INT4 with a level lookup) and at most 8 query heads per KV
// head.  The launchers report the shapes they take (`handled`).
bool fast_format(const kvq_cache_desc* desc, int G) {
  if (G > 8) return false;
  if (desc->nf4) return nf4_table().symmetric;
  return desc->bits == 2 || desc->bits == 4 || desc->bits == 8;
}

cudaError_t launch_decode_fast(const DecodeParams& p, int bits, int gp, cudaStream_t s,
                               bool* handled, int* occ) {
  if (bits == 2) return launch_decode_fast_int2(p, gp, s, handled, occ);
  if (bits == 4) return launch_decode_fast_int4(p, gp, s, handled, occ);
  return launch_decode_fast_int8(p, gp, s, handled, occ);
}

// Which decode kernel runs for a descriptor and query-head count: the
// tensor-core kernel when an instantiation exists, else the generic one.
struct Plan {
  bool fast = false;
  int gp = 1;
  int occ = 0;  // tensor-core kernel: resident CTAs per SM
  int32_t splits = 0;
};

kvq_status make_plan(const kvq_cache_desc* desc, const CacheGeom& geom, int32_t batch,
                     int32_t num_q_heads, int32_t max_seq_len, int32_t requested, Plan* plan) {
  const int G = num_q_heads / desc->num_kv_heads;
  int occ = 0;
  plan->fast = false;
  if (fast_format(desc, G)) {
    int gp = 1;
    while (gp < G) gp <<= 1;
    plan->gp = gp;
    if (requested > 0) {  // no device query: the occupancy is looked up at launch if needed
      plan->splits = choose_splits((int64_t)batch * desc->num_kv_heads, max_seq_len, requested, 0);
      return KVQ_OK;
    }
    DecodeParams probe{};
    probe.geom = geom;
    probe.G = G;
    bool handled = false;
    cudaError_t e = launch_decode_fast(probe, desc->bits, gp, nullptr, &handled, &occ);
    if (handled && e != cudaSuccess) return from_cuda(e);
    plan->fast = handled;
    if (handled) plan->occ = occ;
  }
  if (requested > 0) {
    plan->splits = choose_splits((int64_t)batch * desc->num_kv_heads, max_seq_len, requested, 0);
    return KVQ_OK;
  }
  if (!plan->fast) {
    DecodeParams probe{};
    probe.geom = geom;
    probe.G = G;
    occ = generic_ctas_per_sm(probe);
  }
  plan->splits = choose_splits((int64_t)batch * desc->num_kv_heads, max_seq_len, 0, occ);
  // More units than one wave holds, and the tensor-core kernel takes them
  // longest first: whole sequences in that order balance better than splits
  // of them, which the model above prices as if every sequence were
  // max_seq_len long (the paged small-model batch: 47.8 us with one split,
  // 53.7 us with two).
  if (plan->fast && batch > 1 && batch <= kLongestFirstMaxBatch &&
      (int64_t)batch * desc->num_kv_heads >= (int64_t)sm_count() * occ)
    plan->splits = 1;
  return plan->splits > 0 ? KVQ_OK : KVQ_ERR_CUDA;
}


#ifdef KVQ_DEBUG
// Bytes kvq_debug_shrink_extent takes off each array's extent.
int64_t g_dbg_shrink[KVQ_ARRAY_COUNT] = {};

void dbg_set(DbgExtents& x, int a, const void* base, size_t bytes) {
  const unsigned long long lo = (unsigned long long)reinterpret_cast<uintptr_t>(base);
  const size_t cut = std::min<size_t>((size_t)g_dbg_shrink[a], bytes);
  x.lo[a] = lo;
  x.hi[a] = base ? lo + (bytes - cut) : lo;
}
#endif

// Debug builds: the extent of every caller array of a call (the sizes
// kvq.h states for debug builds); nothing in a release build.
void dbg_fill(CacheGeom& g, const kvq_cache_desc* desc, const kvq_cache* cache, int32_t batch,
              int32_t num_q_heads, int32_t num_new, const void* q, const void* k_new,
              const void* v_new, const void* lens, const void* out, const void* ws,
              size_t ws_bytes, uint32_t* status) {
#ifdef KVQ_DEBUG
  DbgExtents& x = g.dbg;
  memset(&x, 0, sizeof(x));
  size_t cb = 0, hb = 0;
  if (kvq_cache_array_bytes(desc, batch, &cb, &hb) != KVQ_OK) cb = hb = 0;
  const size_t wb = kvq_cache_window_bytes(desc, batch);
  dbg_set(x, KVQ_ARRAY_K_CODES, cache->k_codes, cb);
  dbg_set(x, KVQ_ARRAY_V_CODES, cache->v_codes, cb);
  dbg_set(x, KVQ_ARRAY_K_SCALE, cache->k_scale, hb);
  dbg_set(x, KVQ_ARRAY_K_ZERO, cache->k_zero, hb);
  dbg_set(x, KVQ_ARRAY_V_SCALE, cache->v_scale, hb);
  dbg_set(x, KVQ_ARRAY_V_ZERO, cache->v_zero, hb);
  dbg_set(x, KVQ_ARRAY_K_WINDOW, cache->k_window, wb);
  dbg_set(x, KVQ_ARRAY_V_WINDOW, cache->v_window, wb);
  dbg_set(x, KVQ_ARRAY_BLOCK_TABLE, cache->block_table,
          desc->layout == KVQ_PAGED ? (size_t)batch * desc->max_blocks_per_seq * 4 : 0);
  const size_t qb = (size_t)batch * num_q_heads * desc->head_dim * 2;
  dbg_set(x, KVQ_ARRAY_Q, q, qb);
  dbg_set(x, KVQ_ARRAY_OUT, out, qb);
  const size_t nb = (size_t)batch * num_new * desc->num_kv_heads * desc->head_dim * 2;
  dbg_set(x, KVQ_ARRAY_K_NEW, k_new, nb);
  dbg_set(x, KVQ_ARRAY_V_NEW, v_new, nb);
  dbg_set(x, KVQ_ARRAY_SEQ_LENS, lens, (size_t)batch * 4);
  dbg_set(x, KVQ_ARRAY_WORKSPACE, ws, ws_bytes);
  x.status = status;
#else
  (void)g, (void)desc, (void)cache, (void)batch, (void)num_q_heads, (void)num_new, (void)q;
  (void)k_new, (void)v_new, (void)lens, (void)out, (void)ws, (void)ws_bytes, (void)status;
#endif
}

}  // namespace

size_t workspace_bytes(int64_t batch, int64_t Hq, int64_t D, int64_t splits) {
  if (splits <= 1) return 0;
  const size_t o = (size_t)(batch * Hq * splits * D) * sizeof(float);
  const size_t ml = (size_t)(batch * Hq * splits * 2) * sizeof(float);
  return ((o + 255) & ~(size_t)255) + ml;
}

void workspace_carve(void* ws, int64_t batch, int64_t Hq, int64_t D, int64_t splits,
                     float** ws_o, float** ws_ml) {
  const size_t o = (size_t)(batch * Hq * splits * D) * sizeof(float);
  *ws_o = reinterpret_cast<float*>(ws);
  *ws_ml = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + ((o + 255) & ~(size_t)255));
}

}  // namespace kvq

using namespace kvq;

extern "C" {

size_t kvq_cache_bytes(const kvq_cache_desc* desc, int64_t tokens) {
  CacheGeom g;
  if (check_desc(desc, &g) == KVQ_ERR_INVALID_ARG || tokens < 0) return 0;
  if (g.kch) {
    // fp16 sinks and residual rows (K and V), then per completed block: g
    // code rows of K and V, a K scale + zero per channel, a V scale + zero
    // per group of each token
    const int64_t S = std::min<int64_t>(g.sink, tokens);
    const int64_t nb = (tokens - S) / g.g;
    const int64_t fp16_rows = tokens - nb * g.g;
    const int64_t per_block = 2LL * g.g * g.row_bytes + 4LL * g.D + 4LL * g.g * g.ngroups;
    return (size_t)(g.Hkv * (2LL * 2 * g.D * fp16_rows + nb * per_block));
  }
  const int64_t per_vector =
      g.row_bytes + (g.bits == 16 ? 0 : ((g.sym || g.nf4) ? 2LL : 4LL) * g.ngroups);
  return (size_t)(2LL * g.Hkv * tokens * per_vector);
}

size_t kvq_cache_window_bytes(const kvq_cache_desc* desc, int32_t batch) {
  CacheGeom g;
  if (check_desc(desc, &g) == KVQ_ERR_INVALID_ARG || batch < 0 || !g.kch) return 0;
  return (size_t)batch * g.Hkv * (g.sink + g.g) * g.D * 2;
}

kvq_status kvq_cache_array_bytes(const kvq_cache_desc* desc, int32_t batch,
                                 size_t* codes_bytes, size_t* header_bytes) {
  CacheGeom g;
  const kvq_status st = check_desc(desc, &g);
  if (st != KVQ_OK) return st;
  if (!codes_bytes || !header_bytes) return KVQ_ERR_INVALID_ARG;
  int64_t rows;
  if (g.layout == KVQ_DENSE) {
    if (batch < 0) return KVQ_ERR_INVALID_ARG;
    rows = (int64_t)batch * g.Hkv * g.slots;
  } else {
    rows = (int64_t)g.num_pages * g.Hkv * g.slots;
  }
  *codes_bytes = (size_t)(rows * g.row_bytes);
  *header_bytes = g.bits == 16 ? 0 : (size_t)(rows * g.ngroups * 2);
  return KVQ_OK;
}

kvq_status kvq_append(const kvq_cache_desc* desc, const kvq_cache* cache, int32_t batch,
                      int32_t num_new, const uint16_t* k_new, const uint16_t* v_new,
                      const int32_t* seq_lens_before, uint32_t* dev_status, void* stream) {
  AppendParams p{};
  kvq_status st = check_desc(desc, &p.geom);
  if (st != KVQ_OK) return st;
  if ((st = check_cache(desc, cache)) != KVQ_OK) return st;
  if (batch < 0 || num_new < 0) return KVQ_ERR_INVALID_ARG;
  if (batch == 0 || num_new == 0) return KVQ_OK;
  if (desc->k_per_channel && batch > KVQ_MAX_BATCH) return KVQ_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !seq_lens_before) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_new) || !aligned(v_new) || !aligned(seq_lens_before)) return KVQ_ERR_INVALID_ARG;
  p.geom.block_table = cache->block_table;
  p.codes[0] = reinterpret_cast<uint8_t*>(cache->k_codes);
  p.codes[1] = reinterpret_cast<uint8_t*>(cache->v_codes);
  p.scale[0] = reinterpret_cast<__half*>(cache->k_scale);
  p.scale[1] = reinterpret_cast<__half*>(cache->v_scale);
  p.zero[0] = reinterpret_cast<__half*>(cache->k_zero);
  p.zero[1] = reinterpret_cast<__half*>(cache->v_zero);
  p.src[0] = reinterpret_cast<const __half*>(k_new);
  p.src[1] = reinterpret_cast<const __half*>(v_new);
  p.window[0] = reinterpret_cast<__half*>(cache->k_window);
  p.window[1] = reinterpret_cast<__half*>(cache->v_window);
  if (p.geom.nf4) memcpy(p.nf4_mid, nf4_table().mid, sizeof(p.nf4_mid));
  p.seq_lens_before = seq_lens_before;
  p.status = dev_status;
  p.batch = batch;
  p.num_new = num_new;
  dbg_fill(p.geom, desc, cache, batch, 0, num_new, nullptr, k_new, v_new, seq_lens_before,
           nullptr, nullptr, 0, dev_status);
  return from_cuda(launch_append(p, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvq_decode_num_splits(const kvq_cache_desc* desc, int32_t batch, int32_t num_q_heads,
                              int32_t max_seq_len, int32_t num_splits) {
  CacheGeom g;
  if (check_desc(desc, &g) != KVQ_OK || batch < 0 || num_q_heads <= 0 || max_seq_len < 0 ||
      num_splits < 0 || num_q_heads % desc->num_kv_heads)
    return 0;
  Plan plan;
  if (make_plan(desc, g, batch, num_q_heads, max_seq_len, num_splits, &plan) != KVQ_OK) return 0;
  return plan.splits;
}

size_t kvq_decode_workspace_size(const kvq_cache_desc* desc, int32_t batch, int32_t num_q_heads,
                                 int32_t max_seq_len, int32_t num_splits) {
  const int32_t s = kvq_decode_num_splits(desc, batch, num_q_heads, max_seq_len, num_splits);
  if (s <= 1) return 0;
  return workspace_bytes(batch, num_q_heads, desc->head_dim, s);
}

}  // extern "C"

namespace {

// Validation, planning and dispatch shared by the decode entry points.  With
// lens_before set the new token's K/V are quantized and attended in the same
// pass (fused append); otherwise seq_lens gives the lengths to attend over.
kvq_status decode_impl(const kvq_cache_desc* desc, const kvq_cache* cache, int32_t batch,
                       int32_t num_q_heads, const uint16_t* q, const int32_t* seq_lens,
                       const int32_t* lens_before, const uint16_t* k_new, const uint16_t* v_new,
                       int32_t max_seq_len, int32_t num_splits, float softmax_scale,
                       uint16_t* out, void* workspace, size_t workspace_size,
                       uint32_t* dev_status, void* stream) {
  DecodeParams p{};
  kvq_status st = check_desc(desc, &p.geom);
  if (st != KVQ_OK) return st;
  if ((st = check_cache(desc, cache)) != KVQ_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_seq_len < 0 || num_splits < 0)
    return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % desc->num_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale >= 0.f) || isinf(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if (batch == 0) return KVQ_OK;
  const bool fused = lens_before != nullptr;
  if (!q || !out || (!fused && !seq_lens) || (fused && (!k_new || !v_new)))
    return KVQ_ERR_INVALID_ARG;
  if (!aligned(q) || !aligned(out)) return KVQ_ERR_INVALID_ARG;
  if (fused ? (!aligned(lens_before) || !aligned(k_new) || !aligned(v_new)) : !aligned(seq_lens))
    return KVQ_ERR_INVALID_ARG;
  const int G = num_q_heads / desc->num_kv_heads;
  if (G > kMaxGroupHeads || batch > KVQ_MAX_BATCH) return KVQ_ERR_UNSUPPORTED;

  Plan plan;
  if ((st = make_plan(desc, p.geom, batch, num_q_heads, max_seq_len, num_splits, &plan)) != KVQ_OK)
    return st;
  const int32_t splits = plan.splits;
  const size_t need = workspace_bytes(batch, num_q_heads, desc->head_dim, splits);
  if (need > 0 && (!workspace || workspace_size < need || !aligned(workspace)))
    return KVQ_ERR_WORKSPACE;

  p.geom.block_table = cache->block_table;
  p.codes[0] = reinterpret_cast<const uint8_t*>(cache->k_codes);
  p.codes[1] = reinterpret_cast<const uint8_t*>(cache->v_codes);
  p.scale[0] = reinterpret_cast<const __half*>(cache->k_scale);
  p.scale[1] = reinterpret_cast<const __half*>(cache->v_scale);
  p.zero[0] = reinterpret_cast<const __half*>(cache->k_zero);
  p.zero[1] = reinterpret_cast<const __half*>(cache->v_zero);
  p.q = reinterpret_cast<const __half*>(q);
  p.seq_lens = fused ? nullptr : seq_lens;
  p.lens_before = fused ? lens_before : nullptr;
  p.new_kv[0] = reinterpret_cast<const __half*>(k_new);
  p.new_kv[1] = reinterpret_cast<const __half*>(v_new);
  p.window[0] = reinterpret_cast<const __half*>(cache->k_window);
  p.window[1] = reinterpret_cast<const __half*>(cache->v_window);
  if (p.geom.nf4) memcpy(p.nf4_level, nf4_table().level, sizeof(p.nf4_level));
  p.out = reinterpret_cast<__half*>(out);
  p.ws_o = nullptr;
  p.ws_ml = nullptr;
  if (splits > 1) workspace_carve(workspace, batch, num_q_heads, desc->head_dim, splits, &p.ws_o, &p.ws_ml);
  p.status = dev_status;
  dbg_fill(p.geom, desc, cache, batch, num_q_heads, fused ? 1 : 0, q, k_new, v_new,
           fused ? (const void*)lens_before : (const void*)seq_lens, out,
           splits > 1 ? workspace : nullptr, splits > 1 ? workspace_size : 0, dev_status);
  p.batch = batch;
  p.Hq = num_q_heads;
  p.G = G;
  p.splits = splits;
  p.chunk = split_chunk(max_seq_len, splits);
  // (a paged axis-aware cache pages only the tokens after its sinks)
  const int64_t cap = desc->layout == KVQ_DENSE
                          ? (int64_t)desc->capacity
                          : (int64_t)desc->capacity * desc->max_blocks_per_seq +
                                (desc->k_per_channel ? desc->sink_tokens : 0);
  p.len_limit = (int32_t)std::min<int64_t>(cap, max_seq_len);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)desc->head_dim);
  p.scale_log2 = scale * 1.4426950408889634f;
  // more CTAs than fit at once: start the longest sequences first, so that
  // the last wave holds short ones
  const bool fast_shape = fast_format(desc, G);
  int occ = plan.occ;
  if (fast_shape && occ == 0 && batch > 1 && batch <= kLongestFirstMaxBatch) {
    DecodeParams probe{};
    probe.geom = p.geom;
    probe.G = G;
    bool fast = false;
    const cudaError_t pe = launch_decode_fast(probe, desc->bits, plan.gp, nullptr, &fast, &occ);
    if (fast && pe != cudaSuccess) return from_cuda(pe);
    if (!fast) occ = 0;
  }
  p.rows32 = desc->layout == KVQ_PAGED &&
             (int64_t)desc->num_pages * desc->num_kv_heads * desc->capacity * p.geom.row_bytes <
                 ((int64_t)1 << 31);
  p.longest_first = fast_shape && occ > 0 && batch > 1 && batch <= kLongestFirstMaxBatch &&
                    (int64_t)splits * desc->num_kv_heads * batch > (int64_t)sm_count() * occ;

  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  bool handled = false;
  // the fast kernel appends in-launch for per-token caches; axis-aware
  // caches and shapes without a fast kernel run the append kernels first
  bool appended = false;
  auto append_first = [&]() -> cudaError_t {
    appended = true;
    AppendParams a{};
    a.geom = p.geom;
    a.codes[0] = reinterpret_cast<uint8_t*>(cache->k_codes);
    a.codes[1] = reinterpret_cast<uint8_t*>(cache->v_codes);
    a.scale[0] = reinterpret_cast<__half*>(cache->k_scale);
    a.scale[1] = reinterpret_cast<__half*>(cache->v_scale);
    a.zero[0] = reinterpret_cast<__half*>(cache->k_zero);
    a.zero[1] = reinterpret_cast<__half*>(cache->v_zero);
    a.src[0] = p.new_kv[0];
    a.src[1] = p.new_kv[1];
    a.window[0] = reinterpret_cast<__half*>(cache->k_window);
    a.window[1] = reinterpret_cast<__half*>(cache->v_window);
    if (a.geom.nf4) memcpy(a.nf4_mid, nf4_table().mid, sizeof(a.nf4_mid));
    a.seq_lens_before = lens_before;
    a.status = dev_status;
    a.batch = batch;
    a.num_new = 1;
    return launch_append(a, s);
  };
  // axis-aware caches: with one split the tensor-core kernel appends in its
  // own CTAs (each (sequence, KV head) has one); otherwise, and for shapes
  // it does not take, the append kernel runs first
  if (fused && desc->k_per_channel) {
    if (splits == 1 && fast_shape) p.kch_append = 1;
    else e = append_first();
  }
  if (e == cudaSuccess && fast_format(desc, G)) {
    p.merge_all = splits > 1;
    e = launch_decode_fast(p, desc->bits, plan.gp, s, &handled, nullptr);
  }
  if (e == cudaSuccess && !handled) {
    p.kch_append = 0;
    p.merge_all = 0;
    if (fused && !appended) e = append_first();
    if (e == cudaSuccess) e = launch_decode_generic(p, s);
  }
  if (e == cudaSuccess && splits > 1) e = launch_merge(p, s);
  return from_cuda(e);
}

}  // namespace

extern "C" {

kvq_status kvq_decode_attn(const kvq_cache_desc* desc, const kvq_cache* cache, int32_t batch,
                           int32_t num_q_heads, const uint16_t* q, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t num_splits, float softmax_scale,
                           uint16_t* out, void* workspace, size_t workspace_size,
                           uint32_t* dev_status, void* stream) {
  return decode_impl(desc, cache, batch, num_q_heads, q, seq_lens, nullptr, nullptr, nullptr,
                     max_seq_len, num_splits, softmax_scale, out, workspace, workspace_size,
                     dev_status, stream);
}

kvq_status kvq_append_decode_attn(const kvq_cache_desc* desc, const kvq_cache* cache,
                                  int32_t batch, int32_t num_q_heads, const uint16_t* k_new,
                                  const uint16_t* v_new, const uint16_t* q,
                                  const int32_t* seq_lens_before, int32_t max_seq_len,
                                  int32_t num_splits, float softmax_scale, uint16_t* out,
                                  void* workspace, size_t workspace_size, uint32_t* dev_status,
                                  void* stream) {
  if (batch > 0 && !seq_lens_before) return KVQ_ERR_INVALID_ARG;
  if (batch > 0 && (!k_new || !v_new)) return KVQ_ERR_INVALID_ARG;
  return decode_impl(desc, cache, batch, num_q_heads, q, nullptr, seq_lens_before, k_new, v_new,
                     max_seq_len, num_splits, softmax_scale, out, workspace, workspace_size,
                     dev_status, stream);
}

int32_t kvq_debug_checks(void) {
#ifdef KVQ_DEBUG
  return 1;
#else
  return 0;
#endif
}

kvq_status kvq_debug_shrink_extent(int32_t array, int64_t bytes) {
#ifdef KVQ_DEBUG
  if (array < 0 || array >= KVQ_ARRAY_COUNT || bytes < 0) return KVQ_ERR_INVALID_ARG;
  g_dbg_shrink[array] = bytes;
  return KVQ_OK;
#else
  (void)array, (void)bytes;
  return KVQ_ERR_UNSUPPORTED;
#endif
}

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG: invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED: shape not supported";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE: workspace missing or too small";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA: CUDA runtime error";
  }
  return "KVQ_ERR_UNKNOWN";
}

}  // extern "C"
