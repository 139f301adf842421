// tv_tree_attention_verify_noalloc: the tree-attention call for callers that
// cannot allocate device memory.
//
// tv_tree_attention_verify needs a caller-provided scratch workspace (split-KV
// partial results and arrival counters). Some callers have no way to get one:
// a plugin inside a host framework that only hands over a stream and tensors,
// code running while another component owns the whole device memory pool, or
// a real-time loop that must not call cudaMalloc (it can synchronise the
// device). This entry point takes its scratch from a file-scope __device__
// array instead and allocates nothing.
//
// The array is TV_NOALLOC_SCRATCH_BYTES (64 MiB) per GPU. It belongs to this
// translation unit's module, which the CUDA runtime loads (and so reserves the
// array) the first time the entry point is used on a device; it stays reserved
// until the process exits. The published tree verification methods have no
// counterpart to this call.
#include "tv_common.cuh"

namespace tv {


constexpr size_t kTvNoAllocScratchBytes = TV_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kTvNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device, looked up on the first call
// made with that device current. Host code cannot use the array's name as a
// device pointer: in host code it is only a stand-in for the symbol. Threads
// making their first call at the same time may both look the address up and
// store it; they store the same value, so that race is benign.
static void* g_scratch_addr[kMaxDevices] = {nullptr};

static int scratch_for_current_device(void** out) {
  const int dev = current_device();
  if (dev < 0) return TV_ERR_CUDA;
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return TV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TV_OK;
}

}  // namespace tv

extern "C" int tv_tree_attention_verify_noalloc(
    const tv_geom* geom, int32_t batch, int32_t max_nodes, const void* q, const void* k_new,
    const void* v_new, const int32_t* cu_nodes, const int32_t* positions,
    const uint32_t* mask_bits, const int32_t* prompt_len, const int32_t* block_table,
    const int32_t* n_blocks, int32_t max_blocks_per_req, void* k_cache, void* v_cache,
    int32_t num_blocks, void* out, int32_t* status, void* stream) {
  int rc = tv::check_geom(geom);
  if (rc != TV_OK) return rc;
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES) return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  size_t need = 0;
  rc = tv_workspace_bytes(geom, batch, max_nodes, &need);
  if (rc != TV_OK) return rc;
  if (need > tv::kTvNoAllocScratchBytes) return TV_ERR_WORKSPACE;   // batch or tree too large
  void* scratch = nullptr;
  rc = tv::scratch_for_current_device(&scratch);
  if (rc != TV_OK) return rc;
  // The array keeps whatever the previous call left. Nothing in it has to
  // start at zero: every call writes each scratch record before reading it.
  return tv_tree_attention_verify(geom, batch, max_nodes, q, k_new, v_new, cu_nodes, positions,
                                  mask_bits, prompt_len, block_table, n_blocks,
                                  max_blocks_per_req, k_cache, v_cache, num_blocks, out, scratch,
                                  tv::kTvNoAllocScratchBytes, status, stream);
}
