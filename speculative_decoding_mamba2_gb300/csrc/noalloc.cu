// ssm_tree_verify_noalloc: tree verification for callers that cannot allocate
// device memory.
//
// ssm_tree_verify needs a device workspace that the caller allocates.  Some
// callers have no way to do that: an inference runtime that hands a plugin
// only the tensors of the current op and owns every other byte of device
// memory, an embedding that runs under a fixed memory budget with allocation
// forbidden after start-up, or a host program that links this library through
// the C ABI alone and has no allocator of its own to call.  For them this
// entry point takes its scratch from one array compiled into the library:
// `g_verify_scratch`, SSM_NOALLOC_WORKSPACE_BYTES bytes of device memory that
// every GPU which loads the library holds until the process exits.  The entry
// point itself calls no cudaMalloc, cudaFree or allocating library routine.
//
// On its first call on a device (with that device current) it looks up the
// array's device address with cudaGetSymbolAddress and remembers it; make that
// first call before any stream capture.  Every call shares the one array, so
// calls whose GPU work overlaps (other streams, other host threads) race and
// must be serialised by the caller.  The array keeps whatever the last call
// left; nothing in it has to start at zero, because the prep kernel writes every
// entry the main kernel reads before it is read.
#include <mutex>
#include <string>

#include "common.cuh"

namespace ssmtree {

void set_error(const std::string& msg);

namespace {

static __device__ __align__(256) unsigned char g_verify_scratch[SSM_NOALLOC_WORKSPACE_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace ssmtree

using namespace ssmtree;

extern "C" int ssm_tree_verify_noalloc(const ssm_dims* dims, const ssm_params* prm, int32_t n_seq, int32_t n_nodes,
                                       int32_t max_depth, const ssm_node* layout, const uint16_t* xBC,
                                       const uint16_t* dt, const float* h0, const uint16_t* ring,
                                       const int32_t* ring_head, float* y, int32_t* dev_status, void* stream) {
  const char* fn = "ssm_tree_verify_noalloc";
  // the size check comes first and needs no CUDA call; a shape the library rejects
  // (size 0) is handed to ssm_tree_verify, whose validation reports the exact error
  // before it touches the GPU
  const size_t need = ssm_tree_verify_workspace_size(dims, n_seq, n_nodes, max_depth);
  if (need == 0)
    return ssm_tree_verify(dims, prm, n_seq, n_nodes, max_depth, layout, xBC, dt, h0, ring, ring_head, y, nullptr, 0,
                           dev_status, stream);
  if (need > (size_t)SSM_NOALLOC_WORKSPACE_BYTES) {
    set_error(std::string(fn) + ": this batch needs " + std::to_string(need) + " bytes of scratch, more than the " +
              std::to_string((size_t)SSM_NOALLOC_WORKSPACE_BYTES) +
              " compiled into the library; split the batch or call ssm_tree_verify with a workspace");
    return SSM_ERR_CAPACITY;
  }
  if (n_seq == 0) return ssm_tree_verify(dims, prm, 0, n_nodes, max_depth, layout, xBC, dt, h0, ring, ring_head, y,
                                         nullptr, 0, dev_status, stream);
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    set_error(std::string(fn) + ": cudaGetSymbolAddress of the scratch array failed: " + cudaGetErrorString(e));
    return SSM_ERR_CUDA;
  }
  return ssm_tree_verify(dims, prm, n_seq, n_nodes, max_depth, layout, xBC, dt, h0, ring, ring_head, y, scratch,
                         SSM_NOALLOC_WORKSPACE_BYTES, dev_status, stream);
}
