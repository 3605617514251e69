// C-ABI of libindexer_bwd.so: argument checks, workspace sizing, launches.
// The declarations, with their contracts and sources, are in indexer_bwd.h.
#include <mutex>

#include "indexer_bwd.h"
#include "internal.h"

namespace {

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  unsigned* status = nullptr;  // one device word, allocated once
  // a second stream for work that runs beside the caller's stream within a
  // one-call step (the k copy and the kernel choice, beside the score-grad),
  // at the highest priority; the event that forks it and the one that joins
  // the union pass to the choice
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, sel = nullptr;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

// Current device's info; allocates its status word on first use.
int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return IBWD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return IBWD_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    if (d.supported) {
      if (cudaMalloc(&d.status, sizeof(unsigned)) != cudaSuccess) return IBWD_ERR_CUDA;
      if (cudaMemset(d.status, 0, sizeof(unsigned)) != cudaSuccess) return IBWD_ERR_CUDA;
      int least = 0, greatest = 0;
      if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
          cudaStreamCreateWithPriority(&d.side, cudaStreamNonBlocking, greatest) != cudaSuccess ||
          cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&d.sel, cudaEventDisableTiming) != cudaSuccess)
        return IBWD_ERR_CUDA;
    }
    d.ready = true;
  }
  if (!d.supported) return IBWD_ERR_UNSUPPORTED;
  *out = &d;
  return IBWD_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Non-null, 16-byte aligned and addressable by the device.
bool dev_ptr_ok(const void* p) {
  if (!aligned16(p)) return false;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

bool shape_ok(int B, int S_q, int S_k, int H, int D, int L) {
  if (B < 1 || S_q < 1 || S_k < 1 || L < 1) return false;
  if (H < 1 || H > ibwd::kHP) return false;
  if (D < 8 || D > ibwd::kDP || D % 8 != 0) return false;
  const long long slots = (long long)B * S_q * L;
  if (slots >= (1LL << 31)) return false;
  return true;
}

// dense_or_idx: the sparse variant requires topk_idx (the dense one passes NULL).
int score_grad_common(const float* I, float* A, const int32_t* idx, bool dense_or_idx, int B, int S_q, int S_k,
                      int L, float grad_scale, float* dk, int D, void* stream, int ids_global = 0) {
  if (B < 1 || S_q < 1 || S_k < 1 || L < 1) return IBWD_ERR_INVALID_ARG;
  if ((long long)B * S_q * L >= (1LL << 31)) return IBWD_ERR_UNSUPPORTED;
  if (dk && (D < 1 || (long long)B * S_k * D >= (1LL << 40))) return IBWD_ERR_INVALID_ARG;
  if (!aligned16(I) || !aligned16(A) || (dense_or_idx && !aligned16(idx)) || (dk && !aligned16(dk)))
    return IBWD_ERR_INVALID_ARG;
  DeviceInfo* dv = nullptr;
  int rc = device_info(&dv);
  if (rc) return rc;
  if (!dev_ptr_ok(I) || !dev_ptr_ok(A)) return IBWD_ERR_INVALID_ARG;
  if (idx && !dev_ptr_ok(idx)) return IBWD_ERR_INVALID_ARG;
  if (dk && !dev_ptr_ok(dk)) return IBWD_ERR_INVALID_ARG;
  if (static_cast<const void*>(I) == static_cast<const void*>(A)) return IBWD_ERR_INVALID_ARG;
  ibwd::ScoreGradArgs a{};
  a.index_score = I;
  a.attn_score = A;
  a.idx = idx;
  a.rows = (long long)B * S_q;
  a.L = L;
  a.S_q = S_q;
  a.S_k = S_k;
  a.scale = grad_scale / (float)S_q;
  a.dk_zero = dk;
  a.dk_numel = dk ? (long long)B * S_k * D : 0;
  a.status = dv->status;
  a.num_sms = dv->num_sms;
  a.ids_global = ids_global;
  cudaError_t e = ibwd::launch_score_grad(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? IBWD_OK : IBWD_ERR_CUDA;
}

size_t workspace_common(int B, int S_q, int S_k, int H, int D, int L, int mode, bool dense) {
  if (!shape_ok(B, S_q, S_k, H, D, L) || (mode != IBWD_DK_ATOMIC && mode != IBWD_DK_DETERMINISTIC)) return 0;
  return ibwd::gemm_workspace_layout(B, S_q, S_k, H, D, L, mode == IBWD_DK_DETERMINISTIC, dense).total;
}

// need_idx: the sparse variant requires topk_idx (the dense one passes NULL).
// With I (index_score) given this is the whole backward: the score-grad
// kernel writes dI (from I and the attn_score in the dI buffer) over that
// buffer and zeroes dk in atomic mode, then the gemm stage runs, its kernels
// launched programmatically behind the score-grad (cudnn-frontend #730
// commit list: score-grad and GEMM overlapped through programmatic dependent
// launch); every check of both happens before either is launched.
int gemm_common(const uint16_t* q, const uint16_t* k, const float* w, const float* dI, const int32_t* idx,
                bool need_idx, void* dq, void* dw, float* dk, int B, int S_q, int S_k, int H, int D, int L,
                int mode, void* ws, size_t ws_bytes, void* stream, const float* I = nullptr,
                float grad_scale = 0.f, const ibwd_options* opt = nullptr) {
  if (mode != IBWD_DK_ATOMIC && mode != IBWD_DK_DETERMINISTIC) return IBWD_ERR_INVALID_ARG;
  if (B < 1 || S_q < 1 || S_k < 1 || L < 1 || H < 1 || D < 1) return IBWD_ERR_INVALID_ARG;
  if (!shape_ok(B, S_q, S_k, H, D, L)) return IBWD_ERR_UNSUPPORTED;
  // the key sort keeps one counter per key of a batch in shared memory
  if (mode == IBWD_DK_DETERMINISTIC && S_k > 40960) return IBWD_ERR_UNSUPPORTED;
  const ibwd_options o = opt ? *opt : ibwd_options{};
  if ((o.ids_global != 0 && o.ids_global != 1) || (o.dq_bf16 != 0 && o.dq_bf16 != 1) ||
      (o.dw_bf16 != 0 && o.dw_bf16 != 1))
    return IBWD_ERR_INVALID_ARG;
  // global ids address the flattened [B*S_k] keys with int32
  if (o.ids_global && (long long)B * S_k > 2147483647LL) return IBWD_ERR_UNSUPPORTED;
  if (o.dk_bf16 && !aligned16(o.dk_bf16)) return IBWD_ERR_INVALID_ARG;
  // the logit scale: 0 (unset) or positive and finite
  if (!(o.sm_scale == 0.f || (o.sm_scale > 0.f && o.sm_scale <= 3.4028234663852886e38f)))
    return IBWD_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, w, dI, dq, dw, dk};
  for (const void* p : ptrs)
    if (!aligned16(p)) return IBWD_ERR_INVALID_ARG;
  if (need_idx && !aligned16(idx)) return IBWD_ERR_INVALID_ARG;
  if (I && (!aligned16(I) || static_cast<const void*>(I) == static_cast<const void*>(dI)))
    return IBWD_ERR_INVALID_ARG;
  if (!aligned16(ws)) return IBWD_ERR_WORKSPACE;
  DeviceInfo* dv = nullptr;
  int rc = device_info(&dv);
  if (rc) return rc;
  for (const void* p : ptrs)
    if (!dev_ptr_ok(p)) return IBWD_ERR_INVALID_ARG;
  if (idx && !dev_ptr_ok(idx)) return IBWD_ERR_INVALID_ARG;
  if (I && !dev_ptr_ok(I)) return IBWD_ERR_INVALID_ARG;
  if (o.dk_bf16 && !dev_ptr_ok(o.dk_bf16)) return IBWD_ERR_INVALID_ARG;
  const size_t need = ibwd::gemm_workspace_layout(B, S_q, S_k, H, D, L, mode == IBWD_DK_DETERMINISTIC, !need_idx).total;
  if (!ws || ws_bytes < need || !dev_ptr_ok(ws)) return IBWD_ERR_WORKSPACE;
  ibwd::GemmArgs a{};
  a.q = q;
  a.k = k;
  a.w = w;
  a.dI = dI;
  a.idx = idx;
  a.dq = o.dq_bf16 ? nullptr : static_cast<float*>(dq);
  a.dw = o.dw_bf16 ? nullptr : static_cast<float*>(dw);
  a.dq16 = o.dq_bf16 ? static_cast<uint16_t*>(dq) : nullptr;
  a.dw16 = o.dw_bf16 ? static_cast<uint16_t*>(dw) : nullptr;
  a.dk16 = o.dk_bf16;
  a.ids_global = idx ? o.ids_global : 0;
  a.sm_scale = o.sm_scale == 0.f ? 1.f : o.sm_scale;
  a.dk = dk;
  a.B = B;
  a.S_q = S_q;
  a.S_k = S_k;
  a.H = H;
  a.D = D;
  a.L = L;
  a.deterministic = mode == IBWD_DK_DETERMINISTIC;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  a.status = dv->status;
  a.num_sms = dv->num_sms;
  a.side = dv->side;
  a.ev_fork = dv->fork;
  a.ev_sel = dv->sel;
  if (I) {
    // the gemm stage's work that needs neither dI nor the score-grad's dK
    // zeroing (k copy, kernel choice) starts beside the score-grad
    // on the side stream, after everything queued before this call
    if (cudaEventRecord(dv->fork, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaStreamWaitEvent(dv->side, dv->fork, 0) != cudaSuccess)
      return IBWD_ERR_CUDA;
    a.early_side = 1;
    rc = score_grad_common(I, const_cast<float*>(dI), idx, need_idx, B, S_q, S_k, L, grad_scale,
                           mode == IBWD_DK_ATOMIC ? dk : nullptr, D, stream, a.ids_global);
    if (rc) return rc;
    a.after_score_grad = 1;
  }
  cudaError_t e = ibwd::launch_gemm(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? IBWD_OK : IBWD_ERR_CUDA;
}

}  // namespace

// The forward: index_score from q, k, w (and topk_idx unless dense).
int fwd_common(const uint16_t* q, const uint16_t* k, const float* w, const int32_t* idx, bool need_idx, float* out,
               int B, int S_q, int S_k, int H, int D, int L, void* stream) {
  if (B < 1 || S_q < 1 || S_k < 1 || L < 1 || H < 1 || D < 1) return IBWD_ERR_INVALID_ARG;
  if (!shape_ok(B, S_q, S_k, H, D, L)) return IBWD_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k, w, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return IBWD_ERR_INVALID_ARG;
  if (need_idx && !aligned16(idx)) return IBWD_ERR_INVALID_ARG;
  DeviceInfo* dv = nullptr;
  int rc = device_info(&dv);
  if (rc) return rc;
  for (const void* p : ptrs)
    if (!dev_ptr_ok(p)) return IBWD_ERR_INVALID_ARG;
  if (idx && !dev_ptr_ok(idx)) return IBWD_ERR_INVALID_ARG;
  ibwd::FwdArgs a{};
  a.q = q;
  a.k = k;
  a.w = w;
  a.idx = idx;
  a.out = out;
  a.B = B;
  a.S_q = S_q;
  a.S_k = S_k;
  a.H = H;
  a.D = D;
  a.L = L;
  a.status = dv->status;
  a.num_sms = dv->num_sms;
  cudaError_t e = ibwd::launch_fwd(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? IBWD_OK : IBWD_ERR_CUDA;
}

extern "C" {

int indexer_bwd_score_grad(const float* index_score, float* attn_score, const int32_t* topk_idx, int B,
                           int S_q, int S_k, int topk, float grad_scale, float* dk_to_zero, int D,
                           void* stream) {
  return score_grad_common(index_score, attn_score, topk_idx, true, B, S_q, S_k, topk, grad_scale, dk_to_zero,
                           D, stream);
}

size_t indexer_bwd_gemm_workspace_size(int B, int S_q, int S_k, int H, int D, int topk, int dk_mode) {
  return workspace_common(B, S_q, S_k, H, D, topk, dk_mode, false);
}

int indexer_bwd_gemm(const uint16_t* q, const uint16_t* k, const float* w, const float* dI,
                     const int32_t* topk_idx, float* dq, float* dw, float* dk, int B, int S_q, int S_k, int H,
                     int D, int topk, int dk_mode, void* workspace, size_t workspace_bytes, void* stream) {
  return gemm_common(q, k, w, dI, topk_idx, true, dq, dw, dk, B, S_q, S_k, H, D, topk, dk_mode, workspace,
                     workspace_bytes, stream);
}

int indexer_bwd_dense_score_grad(const float* index_score, float* attn_score, int B, int S, float grad_scale,
                                 float* dk_to_zero, int D, void* stream) {
  return score_grad_common(index_score, attn_score, nullptr, false, B, S, S, S, grad_scale, dk_to_zero, D, stream);
}

size_t indexer_bwd_dense_gemm_workspace_size(int B, int S, int H, int D, int dk_mode) {
  return workspace_common(B, S, S, H, D, S, dk_mode, true);
}

int indexer_bwd_dense_gemm(const uint16_t* q, const uint16_t* k, const float* w, const float* dI, float* dq,
                           float* dw, float* dk, int B, int S, int H, int D, int dk_mode, void* workspace,
                           size_t workspace_bytes, void* stream) {
  return gemm_common(q, k, w, dI, nullptr, false, dq, dw, dk, B, S, S, H, D, S, dk_mode, workspace,
                     workspace_bytes, stream);
}

int indexer_bwd(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score, float* attn_score,
                const int32_t* topk_idx, float* dq, float* dw, float* dk, int B, int S_q, int S_k, int H, int D,
                int topk, float grad_scale, int dk_mode, void* workspace, size_t workspace_bytes, void* stream) {
  if (!index_score || !topk_idx) return IBWD_ERR_INVALID_ARG;
  return gemm_common(q, k, w, attn_score, topk_idx, true, dq, dw, dk, B, S_q, S_k, H, D, topk, dk_mode, workspace,
                     workspace_bytes, stream, index_score, grad_scale);
}

int indexer_bwd_ex(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score,
                   float* attn_score, const int32_t* topk_idx, void* dq, void* dw, float* dk, int B, int S_q,
                   int S_k, int H, int D, int topk, float grad_scale, int dk_mode, const ibwd_options* options,
                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!index_score || !topk_idx) return IBWD_ERR_INVALID_ARG;
  return gemm_common(q, k, w, attn_score, topk_idx, true, dq, dw, dk, B, S_q, S_k, H, D, topk, dk_mode, workspace,
                     workspace_bytes, stream, index_score, grad_scale, options);
}

int indexer_bwd_dense_ex(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score,
                         float* attn_score, void* dq, void* dw, float* dk, int B, int S, int H, int D,
                         float grad_scale, int dk_mode, const ibwd_options* options, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!index_score) return IBWD_ERR_INVALID_ARG;
  return gemm_common(q, k, w, attn_score, nullptr, false, dq, dw, dk, B, S, S, H, D, S, dk_mode, workspace,
                     workspace_bytes, stream, index_score, grad_scale, options);
}

int indexer_bwd_dense(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score,
                      float* attn_score, float* dq, float* dw, float* dk, int B, int S, int H, int D,
                      float grad_scale, int dk_mode, void* workspace, size_t workspace_bytes, void* stream) {
  if (!index_score) return IBWD_ERR_INVALID_ARG;
  return gemm_common(q, k, w, attn_score, nullptr, false, dq, dw, dk, B, S, S, H, D, S, dk_mode, workspace,
                     workspace_bytes, stream, index_score, grad_scale);
}

int indexer_fwd(const uint16_t* q, const uint16_t* k, const float* w, const int32_t* topk_idx, float* index_score,
                int B, int S_q, int S_k, int H, int D, int topk, void* stream) {
  if (!topk_idx) return IBWD_ERR_INVALID_ARG;
  return fwd_common(q, k, w, topk_idx, true, index_score, B, S_q, S_k, H, D, topk, stream);
}

int indexer_fwd_dense(const uint16_t* q, const uint16_t* k, const float* w, float* index_score, int B, int S, int H,
                      int D, void* stream) {
  return fwd_common(q, k, w, nullptr, false, index_score, B, S, S, H, D, S, stream);
}

int indexer_bwd_last_device_status(void* stream) {
  DeviceInfo* dv = nullptr;
  int rc = device_info(&dv);
  if (rc) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return IBWD_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, dv->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return IBWD_ERR_CUDA;
  if (word && cudaMemset(dv->status, 0, sizeof word) != cudaSuccess) return IBWD_ERR_CUDA;
  if (word & 1u) return IBWD_ERR_TIMEOUT;
  if (word & 2u) return IBWD_ERR_RANGE;
  return IBWD_OK;
}

const char* indexer_bwd_status_string(int status) {
  switch (status) {
    case IBWD_OK: return "ok";
    case IBWD_ERR_INVALID_ARG: return "invalid argument (null, misaligned or host pointer, or bad shape)";
    case IBWD_ERR_UNSUPPORTED: return "unsupported device or shape";
    case IBWD_ERR_WORKSPACE: return "workspace missing or too small";
    case IBWD_ERR_CUDA: return "CUDA runtime error";
    case IBWD_ERR_TIMEOUT: return "a kernel wait timed out";
    case IBWD_ERR_RANGE: return "a q or k entry lies outside the fp16 range of the tensor-core operands";
    default: return "unknown status";
  }
}

}  // extern "C"
