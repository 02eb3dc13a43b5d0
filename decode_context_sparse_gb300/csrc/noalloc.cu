// mla_decode_dcp_fused_noalloc: the fused DCP decode for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs inside a host runtime which owns every byte of device
// memory and hands a kernel only its inputs and outputs -- a plugin or custom op of
// another inference engine, a serving loop whose memory is reserved once at start-up,
// or a step being recorded into a CUDA graph, where a cudaMalloc would either be
// refused, break the capture, or synchronise the device in the middle of a decode step.
// Such callers cannot provide the split-KV workspace that mla_decode_dcp_fused asks for.
//
// What it does: the same split-KV SIMT kernel as mla_decode_dcp_fused, but its scratch
// (per-split partial outputs, LSEs and merge tickets) lives in the file-scope device
// array below, of fixed size DCP_NOALLOC_SCRATCH_BYTES.  Every GPU that loads this
// library holds that array until the process exits.  All calls on a device share it
// and it keeps the previous call's contents: each call clears the tickets it uses with
// an asynchronous memset on its stream, and calls whose executions overlap on the GPU
// (two streams, or two host threads) race on the array and give wrong results.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DCP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side name of a
// __device__ array is only a stand-in, so the address is looked up once per device,
// with that device current, and cached.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DCP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DCP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DCP_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DCP_OK;
}

}  // namespace

extern "C" int mla_decode_dcp_fused_noalloc(const dcp_mla_decode_args* args, int32_t dcp,
                                            int32_t interleave, dcp_stream_t stream) {
  using namespace dcp;
  DecodeParams p;
  bool sparse;
  int rc = prepare_decode(args, 1, true, dcp, interleave, p, sparse);
  if (rc != DCP_OK) return rc;
  const size_t cap = (size_t)DCP_NOALLOC_SCRATCH_BYTES;
  // a split count the library chose itself is lowered until its scratch fits the array (one
  // split needs none); only a count the caller asked for is rejected when it does not fit
  if (args->num_splits == 0)
    while (p.num_splits > 1 && simt_workspace_bytes(p.num_units, p.heads, p.num_splits) > cap)
      --p.num_splits;
  const size_t need = simt_workspace_bytes(p.num_units, p.heads, p.num_splits);
  if (need > cap) return DCP_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (need > 0) {
    void* base = nullptr;
    if ((rc = scratch_on_current_device(&base)) != DCP_OK) return rc;
    simt_bind_workspace(p, base);
    const size_t tickets = (size_t)p.num_units * (p.heads / kSimtHeadGroup) * sizeof(unsigned);
    if (cudaMemsetAsync(p.ws_cnt, 0, tickets, st) != cudaSuccess) return DCP_ERR_CUDA;
  }
  return launch_decode_simt(p, args->kv_dtype, true, sparse, st) == cudaSuccess ? DCP_OK
                                                                                : DCP_ERR_CUDA;
}
