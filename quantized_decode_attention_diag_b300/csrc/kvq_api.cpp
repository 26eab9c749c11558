// C ABI of the quantized KV-cache library: argument checks, page geometry,
// split planning, kernel dispatch, and the RateQuant greedy allocator.
#include <cuda_runtime_api.h>

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>

#include "kvq.h"
#include "kvq_internal.h"
#include "kvq_logquant.h"

namespace {

thread_local std::string g_last_error;

kvq_status fail(kvq_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks the geometry fields of the descriptor and the bits of `layer`; fills
// the page geometry.  Does not look at the device pointers.
kvq_status check_geometry(const kvq_cache* c, int layer, kvq::LayerGeom* geom) {
  if (!c) return fail(KVQ_EINVAL, "cache descriptor is NULL");
  if (c->num_layers < 1) return fail(KVQ_EINVAL, "num_layers must be >= 1");
  if (layer < 0 || layer >= c->num_layers)
    return fail(KVQ_EINVAL, "layer %d outside [0, %d)", layer, c->num_layers);
  if (c->num_kv_heads < 1 || c->num_kv_heads > kvq::kMaxHeads)
    return fail(KVQ_EUNSUPPORTED, "num_kv_heads %d outside [1, %d]", c->num_kv_heads,
                kvq::kMaxHeads);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(KVQ_EUNSUPPORTED, "head_dim %d not built (64 or 128)", c->head_dim);
  if (c->page_size != kvq::kPage)
    return fail(KVQ_EUNSUPPORTED, "page_size %d not built (16)", c->page_size);
  if ((c->had_block != 1 && c->had_block != 32 && c->had_block != 64 && c->had_block != 128) ||
      c->had_block > c->head_dim)
    return fail(KVQ_EUNSUPPORTED, "Hadamard block %d not built for head_dim %d (1/32/64/128)",
                c->had_block, c->head_dim);
  if (c->window < 0 || c->window > kvq::kMaxWindow)
    return fail(KVQ_EUNSUPPORTED, "window %d outside [0, %d]", c->window, kvq::kMaxWindow);
  if (c->logquant_w != 0) {
    const int a = kvq::lq_log2(c->logquant_w);
    if (a < 1 || c->logquant_w > 256)
      return fail(KVQ_EUNSUPPORTED, "logquant_w %d is not a power of two in [2, 256]",
                  c->logquant_w);
    if (c->window != 0)
      return fail(KVQ_EINVAL, "logquant_w %d needs window 0 (got %d)", c->logquant_w, c->window);
  }
  if (c->key_per_channel != 0 && c->key_per_channel != 1)
    return fail(KVQ_EINVAL, "key_per_channel must be 0 or 1 (got %d)", c->key_per_channel);
  if (c->key_per_channel && c->logquant_w)
    return fail(KVQ_EUNSUPPORTED, "key_per_channel is not built together with logquant_w");
  if (c->num_pages < 1) return fail(KVQ_EINVAL, "num_pages must be >= 1");
  if (!c->bits_host) return fail(KVQ_EINVAL, "bits_host is NULL");
  kvq::LayerGeom local;
  kvq::LayerGeom* g = geom ? geom : &local;
  std::memset(g, 0, sizeof *g);
  long long off = 0;
  int maxh = 0;
  for (int h = 0; h < c->num_kv_heads; ++h) {
    const int bk = c->bits_host[(layer * c->num_kv_heads + h) * 2 + 0];
    const int bv = c->bits_host[(layer * c->num_kv_heads + h) * 2 + 1];
    for (int b : {bk, bv})
      if (b != 2 && b != 4 && b != 8)
        return fail(KVQ_EUNSUPPORTED, "bits %d of layer %d head %d not built (2, 4, 8)", b,
                    layer, h);
    const int hb = c->key_per_channel
                       ? kvq::kPage * (c->head_dim * (bk + bv) / 8) + 2 * c->head_dim + 4 * kvq::kPage
                       : kvq::kPage * (c->head_dim * (bk + bv) / 8 + 8);
    g->head_off[h] = static_cast<int>(off);
    g->bits[h][0] = static_cast<int8_t>(bk);
    g->bits[h][1] = static_cast<int8_t>(bv);
    off += hb;
    if (hb > maxh) maxh = hb;
  }
  g->page_bytes = off;
  g->max_head_bytes = maxh;
  return KVQ_OK;
}

// The descriptor uses window_bufs: a bf16 window, the LogQuant reserve or the
// key-per-channel ring.
bool uses_ring(const kvq_cache* c) {
  return c->window > 0 || c->logquant_w > 0 || c->key_per_channel;
}

// Rows of the bf16 ring per (sequence, KV head, K|V): R, or R + 16 in the
// key-per-channel mode (the page still being filled waits there).
int ring_rows(const kvq_cache* c) { return c->key_per_channel ? c->window + kvq::kPage : c->window; }

// Decode kernel instantiation: 0 token-wise, 1 LogQuant, 2 key-per-channel.
int decode_mode(const kvq_cache* c) { return c->logquant_w ? 1 : c->key_per_channel ? 2 : 0; }

// check_geometry plus the device pointers of `layer`.
kvq_status check_cache(const kvq_cache* c, int layer, kvq::LayerGeom* geom) {
  const kvq_status st = check_geometry(c, layer, geom);
  if (st != KVQ_OK) return st;
  if (c->launch_flags & ~KVQ_LAUNCH_OVERLAP)
    return fail(KVQ_EINVAL, "launch_flags 0x%x has unknown bits", c->launch_flags);
  if (!c->layer_pools || !c->layer_pools[layer])
    return fail(KVQ_EINVAL, "layer_pools[%d] is NULL", layer);
  if (!aligned(c->layer_pools[layer], 16))
    return fail(KVQ_EINVAL, "layer_pools[%d] is not 16-byte aligned", layer);
  if (uses_ring(c)) {
    if (c->max_batch < 1)
      return fail(KVQ_EINVAL,
                  "max_batch must be >= 1 with a window, a LogQuant reserve or per-channel keys");
    if (!c->window_bufs || !c->window_bufs[layer])
      return fail(KVQ_EINVAL,
                  "window_bufs[%d] is NULL but window = %d, logquant_w = %d, key_per_channel = %d",
                  layer, c->window, c->logquant_w, c->key_per_channel);
    if (!aligned(c->window_bufs[layer], 16))
      return fail(KVQ_EINVAL, "window_bufs[%d] is not 16-byte aligned", layer);
  }
  return KVQ_OK;
}

// log2 of the cycles a decode's main loop waits for a page copy before it
// reports KVQ_DEV_COPY_TIMEOUT: 31 (about a second), or the value of the
// environment variable KVQ_DEBUG_COPY_WAIT_LOG2 (0 .. 31; read once), which
// lets a test make the wait run out on copies that do complete.  A warp that
// gives up still waits, with the full limit, for every copy it issued.
int copy_wait_log2() {
  static const int v = [] {
    const char* e = std::getenv("KVQ_DEBUG_COPY_WAIT_LOG2");
    if (!e || !*e) return 31;
    const long x = std::strtol(e, nullptr, 10);
    return x < 0 ? 0 : x > 31 ? 31 : static_cast<int>(x);
  }();
  return v;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cached[dev] = n;
  }
  return cached[dev];
}

struct Plan {
  int S, NS, pages_per_split, stage_bytes, cluster;
  size_t counter_bytes, bytes;
};

// Resident decode CTAs per SM with `smem` bytes of shared memory (the
// occupancy calculator's answer, cached per size, head_dim and mode: a plan
// asks for one or two sizes, and a model's layers may differ in stage size);
// <= 0 when none fits.
constexpr int kOccupancyCache = 16;
int resident_ctas(const kvq_cache* c, size_t smem) {
  static thread_local int cache_key[kOccupancyCache] = {}, cache_val[kOccupancyCache] = {};
  const int mode = decode_mode(c);
  const int key = (static_cast<int>(smem) * 2 + (c->head_dim == 128)) * 4 + mode + 1;
  for (int i = 0; i < kOccupancyCache; ++i)
    if (cache_key[i] == key) return cache_val[i];
  const int bps = kvq::decode_blocks_per_sm(c->head_dim, smem, mode);
  if (bps > 0) {
    for (int i = kOccupancyCache - 1; i > 0; --i) {
      cache_key[i] = cache_key[i - 1];
      cache_val[i] = cache_val[i - 1];
    }
    cache_key[0] = key;
    cache_val[0] = bps;
  }
  return bps;
}

// Split count for one layer: as many splits per (sequence, KV head) as keep the
// whole grid resident in one wave (CTAs per SM from the occupancy calculator
// for this layer's shared-memory size), at least 8 pages (two per warp) per
// split, at most the kernel's split limit.
kvq_status plan_decode(const kvq_cache* c, const kvq::LayerGeom& g, int B, int max_pages,
                       Plan* pl) {
  const int sms = sm_count();
  if (sms <= 0) return fail(KVQ_ECUDA, "no CUDA device visible");
  kvq::DecodeParams probe;
  std::memset(&probe, 0, sizeof probe);
  probe.stage_bytes = (g.max_head_bytes + 127) / 128 * 128;
  probe.R = ring_rows(c);
  probe.lq_w = c->logquant_w;
  probe.kpc = c->key_per_channel;
  const size_t smem = kvq::decode_smem_bytes(probe, c->head_dim);   // no cluster merge
  const int bps = resident_ctas(c, smem);
  if (bps <= 0)
    return fail(KVQ_ECUDA, "decode kernel cannot be resident with %zu bytes of shared memory",
                smem);
  const long long units = static_cast<long long>(B) * c->num_kv_heads;
  // with a window (a LogQuant reserve, a key-per-channel ring), each unit's
  // window CTA takes one of the wave's slots; the key-per-channel ring of a
  // cache without a window holds at most the 15 rows of the open page, which
  // the last split attends to itself
  int extra = uses_ring(c) && !(c->key_per_channel && c->window == 0) ? 1 : 0;
  const long long slots = static_cast<long long>(sms) * bps / units;   // per unit
  // the LogQuant reserve (up to 3W gathered rows) splits over two or four CTAs
  // when a unit has many slots (few sequences): one CTA alone would end last
  if (c->logquant_w > 0 && slots >= 16) extra = slots >= 32 ? 4 : 2;
  long long s = slots - extra;
  const long long cap = (max_pages + 7) / 8;
  if (s > cap) s = cap;
  if (s > kvq::decode_max_splits()) s = kvq::decode_max_splits();
  if (s < 1) s = 1;
  const int pps = static_cast<int>((max_pages + s - 1) / s);
  pl->S = (max_pages + pps - 1) / pps;
  pl->pages_per_split = pps;
  pl->stage_bytes = probe.stage_bytes;
  pl->NS = pl->S + extra;
  pl->cluster = pl->NS <= kvq::decode_max_cluster() ? 1 : 0;
  if (pl->cluster && pl->NS > 1) {
    // the cluster merge gathers the NS partials in CTA 0's shared memory: it is
    // kept while that leaves the CTAs per SM the split count assumed, else the
    // partials meet in global memory
    probe.cluster = 1;
    probe.NS = pl->NS;
    if (resident_ctas(c, kvq::decode_smem_bytes(probe, c->head_dim)) < bps) pl->cluster = 0;
  }
  pl->counter_bytes = (static_cast<size_t>(units) * 4 + 255) / 256 * 256;
  pl->bytes = pl->counter_bytes + static_cast<size_t>(units) * pl->NS * kvq::kMaxGroup *
                                      (c->head_dim + 2) * sizeof(float);
  return KVQ_OK;
}

}  // namespace

namespace kvq {
kvq_status set_last_error(kvq_status status, const char* message) {
  return fail(status, "%s", message);
}
}  // namespace kvq

namespace {

// check_only: every host check, no launch.
kvq_status decode_impl(const kvq_cache* cache, int layer, const void* K_new, const void* V_new,
                       const void* q, int q_is_fp32, const int32_t* page_table, int max_pages,
                       const int32_t* seq_lens, int B, int Hq, float softmax_scale, float* o,
                       void* workspace, size_t ws_bytes, void* stream, bool check_only = false) {
  kvq::DecodeParams p;
  std::memset(&p, 0, sizeof p);
  kvq_status st = check_cache(cache, layer, &p.geom);
  if (st != KVQ_OK) return st;
  if (B < 1 || max_pages < 1) return fail(KVQ_EINVAL, "B and max_pages must be >= 1");
  if (B > 65535) return fail(KVQ_EUNSUPPORTED, "B %d above the grid limit 65535", B);
  if (!q || !o || !page_table || !seq_lens || !workspace)
    return fail(KVQ_EINVAL, "q, o, page_table, seq_lens and workspace must be non-NULL");
  const bool step = K_new != nullptr || V_new != nullptr;
  if (step && (!K_new || !V_new)) return fail(KVQ_EINVAL, "K_new and V_new must both be non-NULL");
  if (step && (!aligned(K_new, 16) || !aligned(V_new, 16)))
    return fail(KVQ_EINVAL, "K_new and V_new must be 16-byte aligned");
  if (!aligned(q, 4) || !aligned(o, 4) || !aligned(page_table, 4) || !aligned(seq_lens, 4))
    return fail(KVQ_EINVAL, "q, o, page_table and seq_lens must be 4-byte aligned");
  if (!aligned(workspace, 16)) return fail(KVQ_EINVAL, "workspace must be 16-byte aligned");
  const int hkv = cache->num_kv_heads;
  if (Hq < hkv || Hq % hkv) return fail(KVQ_EINVAL, "Hq %d is not a multiple of Hkv %d", Hq, hkv);
  const int G = Hq / hkv;
  if (G != 1 && G != 2 && G != 4)
    return fail(KVQ_EUNSUPPORTED, "GQA group %d not built (1, 2, 4)", G);
  if (uses_ring(cache) && B > cache->max_batch)
    return fail(KVQ_EINVAL, "B %d exceeds the window buffers' max_batch %d", B, cache->max_batch);
  if (step && cache->key_per_channel)
    return fail(KVQ_EINVAL, "key-per-channel decode steps append before the decode");
  if (!std::isfinite(softmax_scale) || softmax_scale < 0.f)
    return fail(KVQ_EINVAL, "softmax_scale must be finite and >= 0");
  Plan pl;
  st = plan_decode(cache, p.geom, B, max_pages, &pl);
  if (st != KVQ_OK) return st;
  if (ws_bytes < pl.bytes)
    return fail(KVQ_EWORKSPACE, "workspace of %zu bytes < %zu required", ws_bytes, pl.bytes);
  const float scale =
      softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(cache->head_dim));
  p.pool = static_cast<const uint8_t*>(cache->layer_pools[layer]);
  p.window = uses_ring(cache) ? static_cast<const uint16_t*>(cache->window_bufs[layer]) : nullptr;
  p.q = q;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.o = o;
  p.counters = static_cast<unsigned int*>(workspace);
  p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.counter_bytes);
  p.status = cache->status_dev;
  p.q_fp32 = q_is_fp32 ? 1 : 0;
  p.max_pages = max_pages;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = hkv;
  p.G = G;
  p.R = ring_rows(cache);
  p.kpc = cache->key_per_channel;
  p.lq_w = cache->logquant_w;
  p.lq_a = cache->logquant_w ? kvq::lq_log2(cache->logquant_w) : 0;
  p.lq_rows = cache->logquant_w ? kvq::lq_rows(cache->logquant_w, p.lq_a) : 0;
  p.num_pages = cache->num_pages;
  p.had_block = cache->had_block;
  p.S = pl.S;
  p.NS = pl.NS;
  p.pages_per_split = pl.pages_per_split;
  p.overlap = (cache->launch_flags & KVQ_LAUNCH_OVERLAP) ? 1 : 0;
  p.cluster = pl.cluster;
  p.stage_bytes = pl.stage_bytes;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_log2 = copy_wait_log2();
  p.step = step ? 1 : 0;
  p.k_new = static_cast<const uint16_t*>(K_new);
  p.v_new = static_cast<const uint16_t*>(V_new);
  if (check_only) return KVQ_OK;
  const cudaError_t e = kvq::launch_decode(p, cache->head_dim, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "decode launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

}  // namespace

extern "C" {

size_t kvq_page_bytes(const kvq_cache* cache, int layer) {
  kvq::LayerGeom g;
  if (check_geometry(cache, layer, &g) != KVQ_OK) return 0;
  return static_cast<size_t>(g.page_bytes);
}

}  // extern "C"

namespace {

// kvq_append; lens_after: seq_lens already count the T_new tokens (a
// key-per-channel decode step).
kvq_status append_impl(const kvq_cache* cache, int layer, const void* K, const void* V,
                       const int32_t* page_table, int max_pages, const int32_t* seq_lens, int B,
                       int T_new, int lens_after, void* stream) {
  kvq::AppendParams p;
  std::memset(&p, 0, sizeof p);
  kvq_status st = check_cache(cache, layer, &p.geom);
  if (st != KVQ_OK) return st;
  if (B < 1) return fail(KVQ_EINVAL, "B must be >= 1");
  if (T_new < 0) return fail(KVQ_EINVAL, "T_new must be >= 0");
  if (T_new == 0) return KVQ_OK;
  if (!K || !V || !page_table || !seq_lens)
    return fail(KVQ_EINVAL, "K, V, page_table and seq_lens must be non-NULL");
  if (!aligned(K, 16) || !aligned(V, 16))
    return fail(KVQ_EINVAL, "K and V must be 16-byte aligned");
  if (!aligned(page_table, 4) || !aligned(seq_lens, 4))
    return fail(KVQ_EINVAL, "page_table and seq_lens must be 4-byte aligned");
  if (max_pages < 1) return fail(KVQ_EINVAL, "max_pages must be >= 1");
  if (static_cast<long long>(B) * T_new > (1ll << 28))
    return fail(KVQ_EINVAL, "B * T_new too large");
  if (uses_ring(cache) && B > cache->max_batch)
    return fail(KVQ_EINVAL, "B %d exceeds the window buffers' max_batch %d", B, cache->max_batch);
  p.K = static_cast<const uint16_t*>(K);
  p.V = static_cast<const uint16_t*>(V);
  p.pool = static_cast<uint8_t*>(cache->layer_pools[layer]);
  p.window = uses_ring(cache) ? static_cast<uint16_t*>(cache->window_bufs[layer]) : nullptr;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.status = cache->status_dev;
  p.max_pages = max_pages;
  p.B = B;
  p.T = T_new;
  p.Hkv = cache->num_kv_heads;
  p.R = ring_rows(cache);
  p.num_pages = cache->num_pages;
  p.warps_per_group = static_cast<int>((static_cast<long long>(B) * T_new + 15) / 16);
  p.div_wpg = kvq::make_fastdiv(static_cast<uint32_t>(p.warps_per_group));
  p.div_T = kvq::make_fastdiv(static_cast<uint32_t>(T_new));
  {
    const long long cap = static_cast<long long>(max_pages) * kvq::kPage;
    p.cap_tokens = cap > INT_MAX ? INT_MAX : static_cast<int>(cap);
  }
  p.lq_w = cache->logquant_w;
  p.lq_a = cache->logquant_w ? kvq::lq_log2(cache->logquant_w) : 0;
  p.lq_rows = cache->logquant_w ? kvq::lq_rows(cache->logquant_w, p.lq_a) : 0;
  p.kpc = cache->key_per_channel;
  p.lens_after = lens_after;
  if (p.kpc) {
    if (B > 65535) return fail(KVQ_EUNSUPPORTED, "B %d above the grid limit 65535", B);
    const cudaError_t e = kvq::launch_kpc_append(p, cache->head_dim, cache->had_block,
                                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(KVQ_ECUDA, "append launch: %s", cudaGetErrorString(e));
    return KVQ_OK;
  }
  cudaError_t e = cudaSuccess;
  if (p.lq_w) e = kvq::launch_lq_carry(p, cache->head_dim, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "LogQuant carry launch: %s", cudaGetErrorString(e));
  e = kvq::launch_append(p, cache->head_dim, cache->had_block, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "append launch: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_append(const kvq_cache* cache, int layer, const void* K, const void* V,
                      const int32_t* page_table, int max_pages, const int32_t* seq_lens, int B,
                      int T_new, void* stream) {
  return append_impl(cache, layer, K, V, page_table, max_pages, seq_lens, B, T_new, 0, stream);
}

int kvq_logquant_rows(int w) {
  const int a = kvq::lq_log2(w);
  if (a < 1 || w > 256) return 0;
  return kvq::lq_rows(w, a);
}

long long kvq_logquant_members(long long n, int w, long long* positions, long long max) {
  const int a = kvq::lq_log2(w);
  if (a < 1 || w > 256 || n < 0) {
    fail(KVQ_EINVAL, "kvq_logquant_members: w %d must be a power of two in [2, 256], n >= 0", w);
    return -1;
  }
  long long count = 0;
  for (long long p = 0; p < n; ++p) {
    if (!kvq::lq_member(p, n, w, a)) continue;
    if (positions && count < max) positions[count] = p;
    ++count;
  }
  return count;
}

size_t kvq_window_bytes(const kvq_cache* cache) {
  if (check_geometry(cache, 0, nullptr) != KVQ_OK) return 0;
  if (cache->max_batch < 1) return 0;
  const size_t per_row = static_cast<size_t>(cache->head_dim) * 2;   // bf16
  const size_t planes = static_cast<size_t>(cache->max_batch) * cache->num_kv_heads * 2;
  if (cache->logquant_w > 0)
    return planes * static_cast<size_t>(kvq_logquant_rows(cache->logquant_w)) * per_row;
  if (cache->window > 0 || cache->key_per_channel)
    return planes * static_cast<size_t>(ring_rows(cache)) * per_row;
  return 0;
}

size_t kvq_decode_workspace_bytes(const kvq_cache* cache, int B, int Hq, int max_pages) {
  if (check_geometry(cache, 0, nullptr) != KVQ_OK) return 0;
  if (B < 1 || max_pages < 1 || Hq < 1) {
    fail(KVQ_EINVAL, "B, Hq and max_pages must be >= 1");
    return 0;
  }
  size_t most = 0;   // enough for every layer
  for (int layer = 0; layer < cache->num_layers; ++layer) {
    kvq::LayerGeom g;
    Plan pl;
    if (check_geometry(cache, layer, &g) != KVQ_OK) return 0;
    if (plan_decode(cache, g, B, max_pages, &pl) != KVQ_OK) return 0;
    if (pl.bytes > most) most = pl.bytes;
  }
  return most;
}

kvq_status kvq_decode_attn(const kvq_cache* cache, int layer, const void* q, int q_is_fp32,
                           const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                           int B, int Hq, float softmax_scale, float* o, void* workspace,
                           size_t ws_bytes, void* stream) {
  return decode_impl(cache, layer, nullptr, nullptr, q, q_is_fp32, page_table, max_pages, seq_lens,
                     B, Hq, softmax_scale, o, workspace, ws_bytes, stream);
}

kvq_status kvq_decode_step(const kvq_cache* cache, int layer, const void* K_new, const void* V_new,
                           const void* q, int q_is_fp32, const int32_t* page_table, int max_pages,
                           const int32_t* seq_lens, int B, int Hq, float softmax_scale, float* o,
                           void* workspace, size_t ws_bytes, void* stream) {
  if (!K_new || !V_new) return fail(KVQ_EINVAL, "K_new and V_new must be non-NULL");
  if (cache && cache->key_per_channel == 1) {
    // the token's page is quantized (once complete) by the append; then the
    // decode, whose arguments are checked before anything is launched
    kvq_status st = decode_impl(cache, layer, nullptr, nullptr, q, q_is_fp32, page_table,
                                max_pages, seq_lens, B, Hq, softmax_scale, o, workspace, ws_bytes,
                                stream, true);
    if (st != KVQ_OK) return st;
    if (!aligned(K_new, 16) || !aligned(V_new, 16))
      return fail(KVQ_EINVAL, "K_new and V_new must be 16-byte aligned");
    st = append_impl(cache, layer, K_new, V_new, page_table, max_pages, seq_lens, B, 1, 1, stream);
    if (st != KVQ_OK) return st;
    return decode_impl(cache, layer, nullptr, nullptr, q, q_is_fp32, page_table, max_pages,
                       seq_lens, B, Hq, softmax_scale, o, workspace, ws_bytes, stream);
  }
  return decode_impl(cache, layer, K_new, V_new, q, q_is_fp32, page_table, max_pages, seq_lens, B,
                     Hq, softmax_scale, o, workspace, ws_bytes, stream);
}

kvq_status kvq_fit_distortion(const double* mse, const int* widths, int n_widths, int n,
                              double* alpha, double* beta) {
  if (n < 0 || n_widths < 1) return fail(KVQ_EINVAL, "n must be >= 0 and n_widths >= 1");
  if (n == 0) return KVQ_OK;
  if (!mse || !widths || !alpha || !beta)
    return fail(KVQ_EINVAL, "mse, widths, alpha and beta must be non-NULL");
  for (int a = 0; a < n_widths; ++a)
    for (int b = a + 1; b < n_widths; ++b)
      if (widths[a] == widths[b]) return fail(KVQ_EINVAL, "width %d repeated", widths[a]);
  for (int i = 0; i < n; ++i) {
    const double* d = mse + static_cast<size_t>(i) * n_widths;
    // least squares of y = ln D against b over the usable widths:
    // y = ln alpha - b ln beta
    double sb = 0.0, sy = 0.0;
    int k = 0, last = -1;
    for (int w = 0; w < n_widths; ++w) {
      if (d[w] > 0.0 && std::isfinite(d[w])) {
        sb += widths[w];
        sy += std::log(d[w]);
        ++k;
        last = w;
      }
    }
    if (k >= 2) {
      const double mb = sb / k, my = sy / k;
      double sxx = 0.0, sxy = 0.0;
      for (int w = 0; w < n_widths; ++w) {
        if (d[w] > 0.0 && std::isfinite(d[w])) {
          const double x = widths[w] - mb;
          sxx += x * x;
          sxy += x * (std::log(d[w]) - my);
        }
      }
      const double ln_beta = -sxy / sxx;
      beta[i] = std::exp(ln_beta);
      alpha[i] = std::exp(my + ln_beta * mb);
    } else {
      // one more bit quarters a uniform quantizer's error
      beta[i] = 4.0;
      alpha[i] = k == 1 ? d[last] * std::pow(4.0, widths[last]) : 0.0;
    }
  }
  return KVQ_OK;
}

kvq_status kvq_alloc_bits(const double* w, const double* beta, int n, long long budget,
                          const uint16_t* allowed_mask, int* bits_out, long long* leftover) {
  if (n < 1 || !w || !beta || !bits_out)
    return fail(KVQ_EINVAL, "n >= 1 and non-NULL w, beta, bits_out required");
  for (int i = 0; i < n; ++i) {
    if (!(std::isfinite(w[i]) && w[i] > 0.0))
      return fail(KVQ_EINVAL, "w[%d] must be finite and > 0", i);
    if (!(std::isfinite(beta[i]) && beta[i] > 1.0))
      return fail(KVQ_EINVAL, "beta[%d] must be finite and > 1", i);
    const unsigned m = allowed_mask ? allowed_mask[i] : 0x114u;  // {2, 4, 8}
    if ((m & 0xfffeu) == 0) return fail(KVQ_EINVAL, "allowed_mask[%d] has no width in 1..15", i);
  }
  auto mask_of = [&](int i) -> unsigned {
    return (allowed_mask ? allowed_mask[i] : 0x114u) & 0xfffeu;
  };
  auto next_allowed = [&](int i, int b) -> int {
    const unsigned m = mask_of(i);
    for (int x = b + 1; x <= 15; ++x)
      if (m & (1u << x)) return x;
    return -1;
  };
  // smallest allowed width of every component
  long long used = 0;
  int* bits = bits_out;
  // work on a local copy so that bits_out stays untouched on KVQ_EBUDGET
  std::string scratch(static_cast<size_t>(n) * sizeof(int), '\0');
  int* cur = reinterpret_cast<int*>(&scratch[0]);
  for (int i = 0; i < n; ++i) {
    const unsigned m = mask_of(i);
    int b = 1;
    while (!(m & (1u << b))) ++b;
    cur[i] = b;
    used += b;
  }
  if (used > budget)
    return fail(KVQ_EBUDGET, "budget %lld below the minimum allocation %lld", budget, used);
  for (;;) {
    int best = -1;
    double best_gain = 0.0;
    for (int i = 0; i < n; ++i) {
      const int nxt = next_allowed(i, cur[i]);
      if (nxt < 0) continue;
      const int cost = nxt - cur[i];
      if (cost > budget - used) continue;
      const double gain = w[i] * (std::pow(beta[i], static_cast<double>(-cur[i])) -
                                  std::pow(beta[i], static_cast<double>(-nxt))) /
                          static_cast<double>(cost);
      if (best < 0 || gain > best_gain) {
        best = i;
        best_gain = gain;
      }
    }
    if (best < 0) break;
    const int nxt = next_allowed(best, cur[best]);
    used += nxt - cur[best];
    cur[best] = nxt;
  }
  std::memcpy(bits, cur, static_cast<size_t>(n) * sizeof(int));
  if (leftover) *leftover = budget - used;
  return KVQ_OK;
}

kvq_status kvq_get_status(const kvq_cache* cache, int* device_status) {
  if (!cache || !cache->status_dev || !device_status)
    return fail(KVQ_EINVAL, "cache, cache->status_dev and device_status must be non-NULL");
  int v = 0;
  const cudaError_t e = cudaMemcpy(&v, cache->status_dev, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "status copy: %s", cudaGetErrorString(e));
  *device_status = v;
  return v ? KVQ_EDEVICE : KVQ_OK;
}

kvq_status kvq_reset_status(const kvq_cache* cache, void* stream) {
  if (!cache || !cache->status_dev)
    return fail(KVQ_EINVAL, "cache and cache->status_dev must be non-NULL");
  const cudaError_t e =
      cudaMemsetAsync(cache->status_dev, 0, sizeof(int), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KVQ_ECUDA, "status reset: %s", cudaGetErrorString(e));
  return KVQ_OK;
}

const char* kvq_last_error(void) { return g_last_error.c_str(); }

const char* kvq_version(void) { return "kvq 0.1 sm_103a"; }

}  // extern "C"
