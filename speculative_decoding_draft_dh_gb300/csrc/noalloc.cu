// Greedy tree acceptance for callers that cannot allocate device memory.
//
// dh_tree_accept needs a scratch buffer (the per-node argmax of the target logits) that the caller
// normally allocates and passes as the workspace.  Some callers have no way to do that: code that
// runs inside a serving engine's step where device allocation is not allowed (cudaMalloc can
// synchronise the whole device and stall every other stream), or a host program that owns no
// device allocator and only receives device pointers from elsewhere.  dh_tree_accept_noalloc
// takes the same inputs and outputs but keeps its scratch in a fixed-size array that lives in the
// library's own device memory (a file-scope __device__ array, loaded with the module), so nothing
// is allocated at call time.
//
// Host code cannot use the array's name as a device address (on the host it names a stand-in
// object), so every call asks the runtime for the array's device address on the current device with
// cudaGetSymbolAddress (a host-side lookup: no allocation, no synchronisation).  Asking on every
// call, rather than caching the address, keeps it right after cudaDeviceReset or a new primary
// context, which load the module again, possibly at another address.  The first call on a device
// may load the module, so it should come before any stream capture.  Every call on a device shares
// the one array: calls whose kernels overlap on the GPU (for example on two streams) race on it and
// must be ordered by the caller.
#include "dh_internal.cuh"

namespace dh {
namespace {

// Per-node argmax scratch: DH_TREE_NOALLOC_MAX_NODES int32 entries (B * N nodes per call).
static __device__ __align__(256) int32_t g_tree_scratch[DH_TREE_NOALLOC_MAX_NODES];

// Device address of g_tree_scratch in the current context; nullptr if the runtime cannot resolve
// the symbol (the failure is recorded for dh_last_error).
int32_t* scratch_address() {
  void* p = nullptr;
  if (note_error(cudaGetSymbolAddress(&p, g_tree_scratch), "cudaGetSymbolAddress(tree scratch)") != cudaSuccess)
    return nullptr;
  return static_cast<int32_t*>(p);
}

}  // namespace
}  // namespace dh

using namespace dh;

extern "C" int dh_tree_accept_noalloc(const void* logits, const int32_t* parent, const int32_t* token, int B, int N,
                                      int vocab, int dtype, int32_t* argmax_out, int32_t* path_out, int32_t* len_out,
                                      int32_t* bonus_out, int32_t* err_out, void* stream) {
  if (B < 0 || N <= 0 || vocab <= 0) return DH_ERR_INVALID_ARG;
  if (dtype != DH_F32 && dtype != DH_BF16) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!logits || !parent || !token || !path_out || !len_out || !bonus_out) return DH_ERR_INVALID_ARG;
  if (N > DH_MAX_TREE_NODES) return DH_ERR_UNSUPPORTED;
  if ((long long)B * N > DH_TREE_NOALLOC_MAX_NODES) {
    note_error(cudaErrorInvalidValue, "dh_tree_accept_noalloc: B * N exceeds DH_TREE_NOALLOC_MAX_NODES");
    return DH_ERR_UNSUPPORTED;
  }
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) || ((long long)vocab * (dtype == DH_BF16 ? 2 : 4)) % 16)
    return DH_ERR_UNSUPPORTED;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  int32_t* scratch = scratch_address();
  if (!scratch) return DH_ERR_CUDA;
  if (note_error(launch_tree(c, logits, parent, token, B, N, vocab, dtype, scratch, argmax_out, path_out, len_out,
                             bonus_out, err_out),
                 "tree (no-alloc)") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}
