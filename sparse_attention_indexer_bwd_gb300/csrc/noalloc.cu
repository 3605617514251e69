// indexer_bwd_gemm_noalloc: the gemm stage (atomic dK) with its scratch
// memory in a fixed array that the library owns, for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the
// backward: code inside a custom allocator or a memory-pool callback (an
// allocation there would re-enter the allocator), runtimes that hand out all
// device memory up front and forbid later allocations, and launch paths that
// must not synchronize the device (cudaMalloc and cudaFree may).  This entry
// point takes only inputs and outputs; the one scratch buffer it needs (a
// row counter and the fp16 copy of k of the per-row gemm kernel) lives in
// the array below, which every GPU that loads the library keeps until the
// process exits.
#include <mutex>

#include "indexer_bwd.h"
#include "internal.h"

namespace {

// Scratch: the per-row kernel's row counter (256 bytes) and the fp16 copy of
// k (256 bytes per key row plus one zero row per batch), so
// B * (S_k + 1) <= kMaxKeyRows.
constexpr long long kMaxKeyRows = 32768;
constexpr size_t kScratchBytes = 256 + (size_t)kMaxKeyRows * 256;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];
// Device status word of these calls (a bounded wait that timed out sets a
// bit).  Zero at module load; cleared only by indexer_bwd_gemm_noalloc_status.
static __device__ __align__(256) unsigned g_status;

struct NoAllocDevice {
  bool ready = false;
  int num_sms = 0;
  void* scratch = nullptr;   // device address of g_scratch on this device
  unsigned* status = nullptr;
};
std::mutex g_na_mu;
NoAllocDevice g_na[64];

// Once per device, with that device current: the arrays' device addresses
// (in host code g_scratch only names a host-side stand-in, never a device
// address) and the kernel's shared-memory attribute.  The address lookup may
// load the library's device module, which allocates the arrays.
int noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IBWD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_na_mu);
  NoAllocDevice& d = g_na[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return IBWD_ERR_CUDA;
    if (!(major == 10 && minor == 3)) return IBWD_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    void* status = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_scratch) != cudaSuccess) return IBWD_ERR_CUDA;
    if (cudaGetSymbolAddress(&status, g_status) != cudaSuccess) return IBWD_ERR_CUDA;
    if (ibwd::prepare_gemm_rows() != cudaSuccess) return IBWD_ERR_CUDA;
    d.scratch = scratch;
    d.status = static_cast<unsigned*>(status);
    d.num_sms = sms;
    d.ready = true;
  }
  *out = &d;
  return IBWD_OK;
}

bool na_aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool na_device_ptr(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" int indexer_bwd_gemm_noalloc_setup(void) {
  NoAllocDevice* dv = nullptr;
  return noalloc_setup(&dv);
}

extern "C" int indexer_bwd_gemm_noalloc(const uint16_t* q, const uint16_t* k, const float* w, const float* dI,
                                        const int32_t* topk_idx, float* dq, float* dw, float* dk, int B, int S_q,
                                        int S_k, int H, int D, int topk, void* stream) {
  if (B < 1 || S_q < 1 || S_k < 1 || topk < 1 || H < 1 || D < 1) return IBWD_ERR_INVALID_ARG;
  if (H > ibwd::kHP || D < 8 || D > ibwd::kDP || D % 8 != 0) return IBWD_ERR_UNSUPPORTED;
  if ((long long)B * S_q * topk >= (1LL << 31)) return IBWD_ERR_UNSUPPORTED;
  // beyond the fixed scratch (checked in 64-bit before any size is formed)
  if ((long long)B * ((long long)S_k + 1) > kMaxKeyRows) return IBWD_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, w, dI, topk_idx, dq, dw, dk};
  for (const void* p : ptrs)
    if (!na_aligned16(p)) return IBWD_ERR_INVALID_ARG;
  NoAllocDevice* dv = nullptr;
  int rc = noalloc_setup(&dv);
  if (rc) return rc;
  for (const void* p : ptrs)
    if (!na_device_ptr(p)) return IBWD_ERR_INVALID_ARG;
  ibwd::GemmArgs a{};
  a.q = q;
  a.k = k;
  a.w = w;
  a.dI = dI;
  a.idx = topk_idx;
  a.dq = dq;
  a.dw = dw;
  a.dk = dk;
  a.B = B;
  a.S_q = S_q;
  a.S_k = S_k;
  a.H = H;
  a.D = D;
  a.L = topk;
  a.ws = dv->scratch;  // fully rewritten by every call before it is read
  a.ws_bytes = kScratchBytes;
  a.status = dv->status;
  a.num_sms = dv->num_sms;
  return ibwd::launch_gemm_rows(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? IBWD_OK : IBWD_ERR_CUDA;
}

extern "C" int indexer_bwd_gemm_noalloc_status(void* stream) {
  NoAllocDevice* dv = nullptr;
  int rc = noalloc_setup(&dv);
  if (rc) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return IBWD_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_status, sizeof word) != cudaSuccess) return IBWD_ERR_CUDA;
  if (word) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess) return IBWD_ERR_CUDA;
  }
  if (word & 1u) return IBWD_ERR_TIMEOUT;
  if (word & 2u) return IBWD_ERR_RANGE;
  return IBWD_OK;
}
