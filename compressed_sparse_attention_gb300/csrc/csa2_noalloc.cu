// csa2_attend_noalloc: the attention step for callers that cannot allocate
// device memory themselves.
//
// Some callers of this library may not call cudaMalloc or any allocating
// routine: a host program that owns every byte of device memory through its
// own pool and forbids outside allocations (an inference server's fixed
// arena, a plugin inside another runtime), or a latency-critical loop that
// must never hit the allocator's implicit synchronisation. csa2_attend needs a
// caller-provided workspace for its split-K partial results; this variant
// keeps those partials in one statically sized device array that belongs to
// the library instead. The array is a file-scope __device__ variable, so the
// CUDA runtime places it once per device when this module is first used on
// that device, and it stays there until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// is only a stand-in symbol): the address is looked up with
// cudaGetSymbolAddress, with the context's device current, by the first call
// of this entry point made with a given context, and kept in that context.
// A context is bound to one device and to the lifetime of the CUDA context it
// was created in, so a context created after a device reset looks the address
// up afresh. That first call should come before any stream capture begins on
// the device.
//
// Every call on a device shares the same array and it keeps the last call's
// contents. Nothing in it has to start at zero (each call writes every
// partial it later reads), but two calls whose work overlaps on the GPU (on
// different streams, without ordering between them) race on the array and
// give wrong results: order such calls on one stream.
#include <cstdio>

#include "ctx.cuh"
#include "launchers.cuh"

// the scratch: split-K partial outputs and (max, sum) pairs of csa2_attend
static __device__ __align__(256) unsigned char g_attend_scratch[CSA2_NOALLOC_SCRATCH_BYTES];

extern "C" csa2_status csa2_attend_noalloc(csa2_ctx* ctx, void* stream, int32_t n_seq, int32_t n_query,
                                           const uint16_t* q, const int64_t* q_pos, const int32_t* seq_of_q,
                                           const void* win_kv, const uint8_t* win_scale, const int64_t* win_off,
                                           const int64_t* win_lo, const void* pool_kv, const uint8_t* pool_scale,
                                           const int64_t* pool_off, const int32_t* topk_idx, const float* sink,
                                           uint16_t* out, float* lse) {
  if (!ctx) return CSA2_ERR_INVALID_ARG;
  ctx->last_launches = 0;
  const size_t need = csa2_attend_workspace_size(ctx, n_query);
  if (need > (size_t)CSA2_NOALLOC_SCRATCH_BYTES) {
    char buf[192];
    std::snprintf(buf, sizeof(buf),
                  "attend_noalloc: %d queries need %zu bytes of scratch, more than the library's fixed %zu "
                  "(use csa2_attend with a workspace)",
                  (int)n_query, need, (size_t)CSA2_NOALLOC_SCRATCH_BYTES);
    ctx->err = buf;
    return CSA2_ERR_WORKSPACE;
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    ctx->err = std::string("attend_noalloc: cudaGetDevice: ") + cudaGetErrorString(e);
    return CSA2_ERR_CUDA;
  }
  if (dev != ctx->device) {
    ctx->err = "attend_noalloc: the context's device must be the current device";
    return CSA2_ERR_INVALID_ARG;
  }
  if (ctx->noalloc_scratch == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attend_scratch);
    if (e != cudaSuccess) {
      ctx->err = std::string("attend_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e);
      return CSA2_ERR_CUDA;
    }
    ctx->noalloc_scratch = p;
  }
  void* scratch = ctx->noalloc_scratch;
  return csa2_attend(ctx, stream, n_seq, n_query, q, q_pos, seq_of_q, win_kv, win_scale, win_off, win_lo, pool_kv,
                     pool_scale, pool_off, topk_idx, sink, out, lse, scratch, (size_t)CSA2_NOALLOC_SCRATCH_BYTES);
}
