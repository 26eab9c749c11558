// Decode attention that allocates nothing: kvq_decode_attn_static().
//
// kvq_decode_attn() needs a caller-provided workspace for its split-K partial
// results and per-(sequence, KV head) tickets.  Some callers cannot provide
// one: a plugin running inside a host process whose device memory is owned and
// budgeted by that process's own allocator (it may not call cudaMalloc, nor
// keep a private buffer behind the allocator's back), or a latency-critical
// serving path that must never reach cudaMalloc / cudaFree because those calls
// can synchronise the whole device.  For them this entry point runs the same
// decode with its scratch taken from kvq_static_workspace, a fixed array that
// the library itself owns.  The caller still passes q, o, the cache, the page
// table and the sequence lengths.
#include <cuda_runtime_api.h>

#include <cstdio>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

// Split-K partials and tickets of kvq_decode_attn_static().  Zero when the
// module loads; every GPU that loads the library holds these bytes until the
// process exits.  All calls share them and they keep the last call's contents.
static __device__ __align__(256) unsigned char kvq_static_workspace[KVQ_STATIC_WORKSPACE_BYTES];

// Device address of kvq_static_workspace on the current device.  In host code
// the array's name is only a stand-in for the symbol, not a device address; the
// address comes from cudaGetSymbolAddress with the device current.  It is
// looked up on every call (a host-side query once the module is loaded), so a
// device reset or a re-created primary context, which may move the array,
// cannot leave a stale pointer behind.
cudaError_t workspace_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, kvq_static_workspace);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_static(const kvq_cache* cache, int layer, const void* q,
                                             int q_is_fp32, const int32_t* page_table,
                                             int max_pages, const int32_t* seq_lens, int B,
                                             int Hq, float softmax_scale, float* o,
                                             void* stream) {
  const size_t need = kvq_decode_workspace_bytes(cache, B, Hq, max_pages);
  if (need == 0) return KVQ_EINVAL;  // the reason is already in kvq_last_error()
  if (need > static_cast<size_t>(KVQ_STATIC_WORKSPACE_BYTES)) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "kvq_decode_attn_static: this decode needs %zu bytes of scratch, more than "
                  "the library's fixed %d bytes; use kvq_decode_attn with a workspace",
                  need, KVQ_STATIC_WORKSPACE_BYTES);
    return kvq::set_last_error(KVQ_EWORKSPACE, msg);
  }
  void* ws = nullptr;
  cudaError_t e = workspace_address(&ws);
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "kvq_decode_attn_static: static workspace address: %s",
                  cudaGetErrorString(e));
    return kvq::set_last_error(KVQ_ECUDA, msg);
  }
  // The tickets (one unsigned int per (sequence, KV head), first in the
  // workspace) must start at zero; the partial results are written before
  // they are read and need no clearing.
  const size_t ticket_bytes = (static_cast<size_t>(B) * cache->num_kv_heads * 4 + 255) / 256 * 256;
  e = cudaMemsetAsync(ws, 0, ticket_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof msg, "kvq_decode_attn_static: clearing tickets: %s",
                  cudaGetErrorString(e));
    return kvq::set_last_error(KVQ_ECUDA, msg);
  }
  return kvq_decode_attn(cache, layer, q, q_is_fp32, page_table, max_pages, seq_lens, B, Hq,
                         softmax_scale, o, ws, static_cast<size_t>(KVQ_STATIC_WORKSPACE_BYTES),
                         stream);
}
