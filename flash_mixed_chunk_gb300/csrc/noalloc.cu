// noalloc.cu -- flash_mca_forward_noalloc: the tensor-core forward pass with
// its workspace taken from a fixed array compiled into the library, for
// callers that cannot allocate device memory themselves.
//
// Who needs this: code that runs where cudaMalloc is not available or not
// allowed -- for example a plugin or callback invoked inside a host that owns
// all device memory and hands out only the tensors it manages, code running
// while another component holds an allocation lock, or a caller that must
// never fail half-way because an allocation could not be satisfied.  Such a
// caller can still pass its inputs and output, but cannot provide the
// scratch (the chunks' local state sums, the segment totals and carries, the
// T rows and a grid counter) that flash_mca_forward asks for.
//
// The scratch is one file-scope __device__ array of FMCA_NOALLOC_SCRATCH_BYTES.
// It belongs to this file's module (which holds no kernel): with the CUDA
// runtime's default lazy module loading a GPU receives it the first time this
// entry point looks its address up there, and with eager loading
// (CUDA_MODULE_LOADING=EAGER) every GPU on which the process creates a
// context does, whichever entry points run.  It stays until the process
// exits (or the context is reset).  All calls on a device share it, so calls
// whose work overlaps on that GPU (for example on two streams) race on it;
// calls queued on one stream are ordered and safe.  The array keeps whatever
// the previous call left in it: the forward pass writes every scratch byte it
// reads before reading it, and the one value that must start at zero (the
// counter of output CTAs that have formed their share of the segment
// carries) is cleared by the first kernel of every call, the walkers, before
// the output kernel passes its grid-dependency wait.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "flash_mca.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)FMCA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol: its device address must be obtained with
// cudaGetSymbolAddress, never taken with & on the host.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct CachedAddress {
  void *ptr = nullptr;
  unsigned long long ctx_id = 0;  // context the address belongs to (0: none)
};
CachedAddress g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique ID of the calling thread's current context (0 when there is none or
// the driver cannot say).  A device reset gives the device a new primary
// context with a new ID, and the module -- with the array -- is loaded anew.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch on the current device, looked up with that
// device current the first time and again whenever the device's context has
// changed since the last lookup.  Returns nullptr on failure.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  CachedAddress &c = g_scratch[dev];
  const unsigned long long id = current_context_id();
  if (c.ptr != nullptr && id != 0 && id == c.ctx_id) return c.ptr;
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();  // do not leave the lookup failure as the sticky last error
    return nullptr;
  }
  c.ptr = ptr;
  c.ctx_id = current_context_id();  // the lookup made the context current if it was not
  return ptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fmca_status flash_mca_forward_noalloc(const void *Z, const void *V, const void *U,
                                                 const float *gamma, const float *beta, void *O,
                                                 int B, int n, int s, int e, int C, int causal,
                                                 fmca_dtype dtype, fmca_stream_t stream) {
  if (B <= 0 || n <= 0 || s <= 0 || e <= 0 || C <= 0) return FMCA_ERR_INVALID_ARG;
  if (dtype != FMCA_F32 && dtype != FMCA_BF16) return FMCA_ERR_INVALID_ARG;
  if (C > n || n % C != 0) return FMCA_ERR_SHAPE;
  if (!Z || !V || !U || !gamma || !beta || !O) return FMCA_ERR_INVALID_ARG;
  if (dtype != FMCA_BF16 || !fmca::tc_supported(B, n, s, e, C)) return FMCA_ERR_UNSUPPORTED;
  if ((int64_t)B * n * (s > e ? s : e) >= ((int64_t)1 << 31)) return FMCA_ERR_UNSUPPORTED;
  if (!aligned16(Z) || !aligned16(V) || !aligned16(U) || !aligned16(O) || !aligned16(gamma) ||
      !aligned16(beta))
    return FMCA_ERR_ALIGN;
  // the problem's scratch must fit in the fixed array
  if (fmca::tc_layout(B, n, s, e, C, causal ? 1 : 0, false).total > kNoAllocScratchBytes)
    return FMCA_ERR_WORKSPACE;
  void *scratch = scratch_on_current_device();
  if (scratch == nullptr) return FMCA_ERR_CUDA;
  const int rc = fmca::launch_tc_forward(Z, V, U, gamma, beta, O, B, n, s, e, C, causal ? 1 : 0,
                                         fmca::default_variant(C), scratch,
                                         reinterpret_cast<cudaStream_t>(stream));
  return rc == 0 ? FMCA_OK : FMCA_ERR_CUDA;
}
