// C entry points of libtreeverify that are not tied to one kernel file:
// workspace sizing, the attention entry point's argument checks and launch,
// status names and the interface version.
#include "tv_common.cuh"

namespace tv {
size_t tc_workspace_bytes(int batch, int hq, int hkv, int max_nodes, int head_dim, int grid);
int tc_grid();
int launch_attention_tc(const tv_geom* geom, int batch, int max_nodes, const void* q,
                        const void* k_new, const void* v_new, const int32_t* cu_nodes,
                        const int32_t* positions, const uint32_t* mask, const int32_t* prompt_len,
                        const int32_t* block_table, const int32_t* n_blocks, int max_blocks,
                        void* k_cache, void* v_cache, int num_blocks, void* out, void* workspace,
                        size_t ws_bytes, int32_t* status, cudaStream_t stream);

static int check_device() {
  const int dev = current_device();
  if (dev < 0) return TV_ERR_CUDA;
  const int ok = device_is_sm103(dev);
  if (ok < 0) return TV_ERR_CUDA;
  return ok ? TV_OK : TV_ERR_DEVICE;
}
}  // namespace tv

extern "C" int tv_version(void) { return 4; }

extern "C" int tv_workspace_bytes(const tv_geom* geom, int32_t batch, int32_t max_nodes,
                                  size_t* bytes) {
  int rc = tv::check_geom(geom);
  if (rc != TV_OK) return rc;
  if (bytes == nullptr) return TV_ERR_NULL_POINTER;
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES) return TV_ERR_BAD_SIZE;
  const int grid = tv::tc_grid();
  if (grid <= 0) return TV_ERR_CUDA;
  *bytes = tv::tc_workspace_bytes(batch, geom->num_q_heads, geom->num_kv_heads, max_nodes,
                                  geom->head_dim, grid);
  return TV_OK;
}

extern "C" int tv_tree_attention_verify(const tv_geom* geom, int32_t batch, int32_t max_nodes,
                                        const void* q, const void* k_new, const void* v_new,
                                        const int32_t* cu_nodes, const int32_t* positions,
                                        const uint32_t* mask_bits, const int32_t* prompt_len,
                                        const int32_t* block_table, const int32_t* n_blocks,
                                        int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                                        int32_t num_blocks, void* out, void* workspace,
                                        size_t workspace_bytes, int32_t* status, void* stream) {
  int rc = tv::check_geom(geom);
  if (rc != TV_OK) return rc;
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES || max_blocks_per_req < 1 ||
      num_blocks < 1 || batch > 4096)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!q || !k_new || !v_new || !cu_nodes || !positions || !mask_bits || !prompt_len ||
      !block_table || !n_blocks || !k_cache || !v_cache || !out || !workspace || !status)
    return TV_ERR_NULL_POINTER;
  if (!tv::aligned(q, 16) || !tv::aligned(k_new, 16) || !tv::aligned(v_new, 16) ||
      !tv::aligned(k_cache, 16) || !tv::aligned(v_cache, 16) || !tv::aligned(out, 16) ||
      !tv::aligned(workspace, 256))
    return TV_ERR_MISALIGNED;
  rc = tv::check_device();
  if (rc != TV_OK) return rc;
  return tv::launch_attention_tc(geom, batch, max_nodes, q, k_new, v_new, cu_nodes, positions,
                                 mask_bits, prompt_len, block_table, n_blocks, max_blocks_per_req,
                                 k_cache, v_cache, num_blocks, out, workspace, workspace_bytes,
                                 status, tv::as_stream(stream));
}

extern "C" const char* tv_status_string(int code) {
  switch (code) {
    case TV_OK: return "TV_OK";
    case TV_ERR_NULL_POINTER: return "TV_ERR_NULL_POINTER";
    case TV_ERR_BAD_GEOMETRY: return "TV_ERR_BAD_GEOMETRY";
    case TV_ERR_BAD_SIZE: return "TV_ERR_BAD_SIZE";
    case TV_ERR_WORKSPACE: return "TV_ERR_WORKSPACE";
    case TV_ERR_MISALIGNED: return "TV_ERR_MISALIGNED";
    case TV_ERR_CUDA: return "TV_ERR_CUDA";
    case TV_ERR_DEVICE: return "TV_ERR_DEVICE";
    case TV_ST_BAD_SIZE: return "TV_ST_BAD_SIZE";
    case TV_ST_BAD_ROOT: return "TV_ST_BAD_ROOT";
    case TV_ST_BAD_PARENT: return "TV_ST_BAD_PARENT";
    case TV_ST_BAD_BLOCK: return "TV_ST_BAD_BLOCK";
    case TV_ST_PATH_OVERFLOW: return "TV_ST_PATH_OVERFLOW";
    case TV_ST_TIMEOUT: return "TV_ST_TIMEOUT";
    case TV_ST_BAD_TEMPERATURE: return "TV_ST_BAD_TEMPERATURE";
    default: return "unknown";
  }
}
