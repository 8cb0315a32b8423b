// api.cu -- the C ABI (include/attn_train.h): argument validation, TMA tensor
// maps, workspace carving, launch sequencing and error reporting.  Validation
// runs entirely on the host before anything is enqueued; an unsupported or
// malformed call returns a status and never falls back to another path
// (HOT-Step flash-attn-training, section 2: a silent fallback cannot be told
// apart from a working kernel, so unsupported shapes must fail hard).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "abi_internal.h"
#include "attn_train.h"
#include "kernels.h"
#include "ptx.cuh"

namespace {

using attn::Ctl;
using attn::Dims;
using attn::View;

thread_local char g_msg[512] = "";

attn_status fail(attn_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

attn_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::atomic<uint64_t> g_budget_ns{2000000000ull};

// ATTN_TRAIN_NVTX=1 (read once per process): every entry point that enqueues
// kernels wraps each of its launches in an NVTX range named after the kernel
// pass, for profilers' timelines.  Off by default; then a range costs one
// branch on a cached flag.
bool nvtx_on() {
  static const bool on = [] {
    const char* e = std::getenv("ATTN_TRAIN_NVTX");
    return e != nullptr && e[0] == '1';
  }();
  return on;
}

struct NvtxRange {
  bool on;
  explicit NvtxRange(const char* name) : on(nvtx_on()) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
};

// ----------------------------------------------------- device error word
__device__ uint32_t g_device_error;

constexpr int kMaxDevices = 64;
uint32_t* g_err_ptr[kMaxDevices] = {};
std::mutex g_err_mu;

attn_status device_error_word(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_err_ptr[dev];
  return ATTN_OK;
}

// ------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

attn_status get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (g_encode == nullptr)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)",
                cudaGetErrorString(g_encode_err));
  *fn = g_encode;
  return ATTN_OK;
}

// 4-D map over a [B, H, S, D] bf16 view; box = [128 rows x min(D, 64) cols].
attn_status make_map(CUtensorMap* m, const View& v, int B, int H, int S, int D, const char* name) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  attn_status st = get_encode(&enc);
  if (st != ATTN_OK) return st;
  const int64_t sS = v.ss * 2;
  const int64_t sH = (H > 1 ? v.sh : v.ss * S) * 2;
  const int64_t sB = (B > 1 ? v.sb : sH / 2 * H) * 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)sS, (cuuint64_t)sH, (cuuint64_t)sB};
  const int boxc = D >= 64 ? 64 : D;
  cuuint32_t box[4] = {(cuuint32_t)boxc, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = D >= 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                : D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                          : CU_TENSOR_MAP_SWIZZLE_32B;
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v.ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "tensor map for %s failed (CUresult %d)", name, (int)r);
  return ATTN_OK;
}

// ------------------------------------------------------------ validation
attn_status check_problem(const attn_problem* p) {
  if (p == nullptr) return fail(ATTN_ERR_INVALID, "problem is NULL");
  if (p->B <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Sq <= 0 || p->Skv <= 0 || p->D <= 0)
    return fail(ATTN_ERR_INVALID, "sizes must be positive (B=%d Hq=%d Hkv=%d Sq=%d Skv=%d D=%d)",
                p->B, p->Hq, p->Hkv, p->Sq, p->Skv, p->D);
  if (p->Hq % p->Hkv != 0)
    return fail(ATTN_ERR_INVALID, "Hq (%d) must be a multiple of Hkv (%d)", p->Hq, p->Hkv);
  // the mask arithmetic takes 2^30 as an unbounded extent
  if (p->Sq >= (1 << 30) || p->Skv >= (1 << 30))
    return fail(ATTN_ERR_UNSUPPORTED, "sequence lengths must be below 2^30 (Sq=%d Skv=%d)",
                p->Sq, p->Skv);
  if (p->D != 16 && p->D != 32 && p->D != 64 && p->D != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "head dim %d unsupported (16, 32, 64, 128)", p->D);
  if (p->mask != ATTN_MASK_FULL && p->mask != ATTN_MASK_CAUSAL && p->mask != ATTN_MASK_TTT &&
      p->mask != ATTN_MASK_WINDOW)
    return fail(ATTN_ERR_UNSUPPORTED, "unknown mask kind %d", p->mask);
  if (p->mask == ATTN_MASK_WINDOW) {
    if (p->window_left < 0 || p->window_right < 0)
      return fail(ATTN_ERR_INVALID, "window extents (%d, %d) must be >= 0", p->window_left,
                  p->window_right);
  } else if (p->window_left != 0 || p->window_right != 0) {
    return fail(ATTN_ERR_INVALID, "window extents are set but the mask is not ATTN_MASK_WINDOW");
  }
  if (reinterpret_cast<uintptr_t>(p->seq_lengths) % 4 != 0)
    return fail(ATTN_ERR_ALIGNMENT, "seq_lengths is not 4-byte aligned");
  if (p->add_mask != nullptr) {
    if (p->mask == ATTN_MASK_TTT)
      return fail(ATTN_ERR_UNSUPPORTED, "an additive mask does not combine with the TTT mask");
    if (reinterpret_cast<uintptr_t>(p->add_mask) % 16 != 0)
      return fail(ATTN_ERR_ALIGNMENT, "add_mask is not 16-byte aligned");
    if (p->add_mask_sb < 0 || p->add_mask_sq < p->Skv)
      return fail(ATTN_ERR_INVALID, "add_mask strides: sb >= 0 and sq >= Skv required");
    if (p->add_mask_sb % 8 != 0 || p->add_mask_sq % 8 != 0)
      return fail(ATTN_ERR_ALIGNMENT, "add_mask strides must be multiples of 8 elements");
  }
  if (p->mask == ATTN_MASK_TTT) {
    if (p->ttt_step < 0) return fail(ATTN_ERR_INVALID, "ttt_step %d < 0", p->ttt_step);
    if ((int64_t)p->Skv != (int64_t)(p->ttt_step + 1) * p->Sq)
      return fail(ATTN_ERR_INVALID, "TTT step %d needs Skv == (t+1)*Sq = %lld, got %d",
                  p->ttt_step, (long long)(p->ttt_step + 1) * p->Sq, p->Skv);
  }
  if (!std::isfinite(p->scale)) return fail(ATTN_ERR_INVALID, "scale is not finite");
  if (p->out_dtype != ATTN_OUT_BF16 && p->out_dtype != ATTN_OUT_F32)
    return fail(ATTN_ERR_UNSUPPORTED, "unknown out_dtype %d", p->out_dtype);
  // launch limits: tile grids, the row-wise passes (at least 16 rows per block
  // for the Delta prep, 8 key rows for the TTT suffix pass) and the additive
  // mask's transpose (grid y = query columns / 64, z = batch entries)
  const int64_t grid_q = (int64_t)((p->Sq + 127) / 128) * p->B * p->Hq;
  const int64_t grid_k = (int64_t)((p->Skv + 127) / 128) * p->B * p->Hkv;
  const int64_t rows = (int64_t)p->B * p->Hq * p->Sq;
  const int64_t suffix_rows = (int64_t)p->B * p->Hkv * p->Sq;
  if (grid_q > 0x7fffffffLL || grid_k > 0x7fffffffLL || rows / 16 >= 0x7fffffffLL ||
      suffix_rows / 8 >= 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "problem too large for one launch");
  if (p->add_mask != nullptr && ((int64_t)p->Sq + 7) / 8 * 8 > 64LL * 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "additive mask with Sq = %d above %lld", p->Sq,
                64LL * 65535 - 7);
  if (p->add_mask != nullptr && p->add_mask_sb != 0 && p->B > 65535)
    return fail(ATTN_ERR_UNSUPPORTED, "per-batch additive mask with B = %d above 65535", p->B);
  return ATTN_OK;
}

// esize: element size in bytes (2 for bf16 inputs and bf16 outputs, 4 for fp32 outputs)
attn_status check_tensor(const attn_tensor& t, int B, int H, int S, int D, const char* name,
                         int esize = 2) {
  if (t.ptr == nullptr) return fail(ATTN_ERR_INVALID, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(t.ptr) % 16 != 0)
    return fail(ATTN_ERR_ALIGNMENT, "%s pointer is not 16-byte aligned", name);
  const int64_t strides[3] = {t.stride_b, t.stride_h, t.stride_s};
  const int sizes[3] = {B, H, S};
  const char* names[3] = {"stride_b", "stride_h", "stride_s"};
  for (int i = 0; i < 3; ++i) {
    if (sizes[i] == 1 && i < 2) continue;  // stride of a size-1 dim is never used
    if (strides[i] <= 0) return fail(ATTN_ERR_INVALID, "%s.%s must be positive", name, names[i]);
    if ((strides[i] * esize) % 16 != 0)
      return fail(ATTN_ERR_ALIGNMENT, "%s.%s * %d bytes is not a multiple of 16", name, names[i],
                  esize);
    if (strides[i] * esize >= (int64_t)1 << 40)
      return fail(ATTN_ERR_UNSUPPORTED, "%s.%s too large", name, names[i]);
  }
  if (t.stride_s < D) return fail(ATTN_ERR_INVALID, "%s rows overlap (stride_s < D)", name);
  return ATTN_OK;
}

Dims make_dims(const attn_problem* p) {
  Dims d;
  d.B = p->B;
  d.Hq = p->Hq;
  d.Hkv = p->Hkv;
  d.Sq = p->Sq;
  d.Skv = p->Skv;
  d.D = p->D;
  d.G = p->Hq / p->Hkv;
  d.geom = attn::make_geom(p->mask, p->mask == ATTN_MASK_TTT ? p->ttt_step : 0, p->window_left,
                           p->window_right, p->Sq, p->Skv);
  d.seqlens = p->seq_lengths;
  d.addm = static_cast<const uint16_t*>(p->add_mask);
  d.addm_sb = p->add_mask_sb;
  d.addm_sq = p->add_mask_sq;
  d.scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt((float)p->D);
  d.scale_log2 = d.scale * 1.4426950408889634f;
  d.out_f32 = p->out_dtype == ATTN_OUT_F32 ? 1 : 0;
  return d;
}

View to_view(const attn_tensor& t) {
  View v;
  v.ptr = const_cast<void*>(t.ptr);
  v.sb = t.stride_b;
  v.sh = t.stride_h;
  v.ss = t.stride_s;
  return v;
}

// Workspace: Delta [B, Hq, Sq] fp32, then for TTT steps t > 0 the per-row
// suffix-diagonal weights p and score gradients ds, [B, Hq, Sq, t] fp32 each.
size_t ws_round(size_t n) { return (n + 255) & ~(size_t)255; }
size_t ws_delta_bytes(const attn_problem* p) {
  return ws_round((size_t)p->B * p->Hq * p->Sq * sizeof(float));
}
size_t ws_diag_bytes(const attn_problem* p) {
  const int t = p->mask == ATTN_MASK_TTT ? p->ttt_step : 0;
  return ws_round((size_t)p->B * p->Hq * p->Sq * (size_t)t * sizeof(float));
}
// The additive mask transposed for the dK/dV pass: [Bm][Skv][SqT] bf16 with
// SqT = Sq rounded up to 8 (16-byte rows), Bm = 1 for a mask shared by every
// batch entry, else B.
int64_t mask_t_sq(const attn_problem* p) { return ((int64_t)p->Sq + 7) & ~(int64_t)7; }
size_t ws_mask_t_bytes(const attn_problem* p) {
  if (p->add_mask == nullptr) return 0;
  const size_t bm = p->add_mask_sb == 0 ? 1 : (size_t)p->B;
  return ws_round(bm * (size_t)p->Skv * (size_t)mask_t_sq(p) * 2);
}
size_t ws_bytes_for(const attn_problem* p) {
  return ws_delta_bytes(p) + 2 * ws_diag_bytes(p) + ws_mask_t_bytes(p);
}

// ------------------------------------------- built-in scratch (no-alloc bwd)
// Scratch for attn_train_bwd_noalloc: the backward's whole workspace
// (ws_bytes_for: Delta, B * Hq * Sq floats; at TTT step t also 2 t floats per
// row for the suffix diagonals; with an additive mask its bf16 transpose) must
// fit in 4 MiB.  That is 1,048,576 rows without TTT diagonals or mask (the long
// GQA workload needs 524,288) and about 1,048,576 / (1 + 2t) rows at TTT step t.
// It lives in the module image, so every GPU that loads this library holds it
// until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device.  In host code
// `g_noalloc_scratch` names a host-side shadow, not device memory, so the
// address must come from cudaGetSymbolAddress, once per device.
attn_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(built-in scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}

}  // namespace

namespace attn {
int set_last_error(int status, const char* msg) {
  return fail(static_cast<attn_status>(status), "%s", msg);
}
}  // namespace attn

extern "C" {

attn_status attn_train_supports(const attn_problem* p) {
  attn_status st = check_problem(p);
  if (st == ATTN_OK) g_msg[0] = '\0';
  return st;
}

attn_status attn_train_workspace_size(const attn_problem* p, size_t* bytes) {
  attn_status st = check_problem(p);
  if (st != ATTN_OK) return st;
  if (bytes == nullptr) return fail(ATTN_ERR_INVALID, "bytes is NULL");
  *bytes = ws_bytes_for(p);
  return ATTN_OK;
}

attn_status attn_train_fwd(const attn_problem* p, attn_tensor q, attn_tensor k, attn_tensor v,
                           attn_tensor o, float* lse, void* stream) {
  return attn_train_fwd_ws(p, q, k, v, o, lse, nullptr, 0, stream);
}

attn_status attn_train_fwd_workspace_size(const attn_problem* p, size_t* bytes) {
  attn_status st = check_problem(p);
  if (st != ATTN_OK) return st;
  if (bytes == nullptr) return fail(ATTN_ERR_INVALID, "bytes is NULL");
  *bytes = attn::fwd_split_plan(make_dims(p)).bytes();
  return ATTN_OK;
}

attn_status attn_train_fwd_ws(const attn_problem* p, attn_tensor q, attn_tensor k, attn_tensor v,
                              attn_tensor o, float* lse, void* workspace, size_t ws_bytes,
                              void* stream) {
  attn_status st = check_problem(p);
  if (st != ATTN_OK) return st;
  const int split = workspace != nullptr ? attn::fwd_split_plan(make_dims(p)).split : 0;
  return attn::fwd_with_split(p, split, q, k, v, o, lse, workspace, ws_bytes, stream);
}

attn_status attn_train_describe(const attn_problem* p, char* buf, size_t buf_len, size_t* needed) {
  attn_status st = check_problem(p);
  if (st != ATTN_OK) return st;
  const Dims d = make_dims(p);
  const int D = d.D;
  const int W = needs_general_mask(d) ? 1 : 0;
  const int M = d.addm != nullptr ? 1 : 0;
  const int t = d.geom.ttt;
  const attn::FwdSplit sp = attn::fwd_split_plan(d);
  const attn::FwdShape fs = attn::fwd_shape(d);
  const attn::BwdShape bs = attn::bwd_shape(D);
  const int64_t n_qp = (p->Sq + 2 * attn::kBM - 1) / (2 * attn::kBM);
  const int64_t fwd_ctas = n_qp * p->B * p->Hq * (sp.split > 0 ? sp.nchunk : 1);
  const int64_t dkdv_ctas = (int64_t)((d.geom.kv_main + attn::kBN - 1) / attn::kBN) * p->B * p->Hkv;
  const int64_t dq_ctas = (int64_t)((p->Sq + attn::kBM - 1) / attn::kBM) * p->B * p->Hq;
  const char* mask = p->mask == ATTN_MASK_FULL     ? "full"
                     : p->mask == ATTN_MASK_CAUSAL ? "causal"
                     : p->mask == ATTN_MASK_TTT    ? "ttt"
                                                   : "window";
  const int ch = t <= 1 ? 1 : t <= 2 ? 2 : t <= 4 ? 4 : 8;
  char out[2048];
  int n = snprintf(
      out, sizeof(out),
      "{\"head_dim\":%d,\"mask\":\"%s\",\"ttt_step\":%d,\"general_mask\":%s,"
      "\"additive_mask\":%s,\"outputs\":\"%s\","
      "\"fwd\":{\"kernel\":\"fwd_kernel<%d,%d,%d,%d>\",\"rows_per_cta\":%d,"
      "\"keys_per_tile\":%d,\"ctas\":%lld,\"kv_ring\":%d,\"score_buffers\":%d,"
      "\"smem_bytes\":%d,\"split_key_tiles\":%d,\"split_chunks\":%d,"
      "\"merge_pass\":%s,\"ttt_scores_prepass\":%s},"
      "\"bwd_prep\":{\"kernel\":\"bwd_prep_kernel<%d,%d>\",\"rows\":%lld},"
      "\"bwd_dkdv\":{\"kernel\":\"bwd_dkdv_kernel<%d,%d,%d>\",\"keys_per_cta\":%d,"
      "\"queries_per_tile\":%d,\"ctas\":%lld,\"q_do_stages\":%d,\"smem_bytes\":%d},"
      "\"bwd_dq\":{\"kernel\":\"bwd_dq_kernel<%d,%d,%d>\",\"rows_per_cta\":%d,"
      "\"keys_per_tile\":%d,\"ctas\":%lld,\"k_ring\":%d,\"v_ring\":%d,\"smem_bytes\":%d}",
      D, mask, t, W ? "true" : "false", M ? "true" : "false",
      d.out_f32 ? "fp32" : "bf16", D, W, M, sp.split > 0 ? 1 : 0, 2 * attn::kBM, attn::kBN,
      (long long)fwd_ctas, fs.ring, fs.three_buffers ? 3 : 2, fs.smem, sp.split, sp.nchunk,
      sp.split > 0 ? "true" : "false",
      (t > 0 && t * 4 <= D * (d.out_f32 ? 4 : 2)) ? "true" : "false", D, t > 0 ? 1 : 0,
      (long long)p->B * p->Hq * p->Sq, D, W, M, attn::kBN, attn::kBM, (long long)dkdv_ctas,
      bs.dkdv_stages, bs.dkdv_smem, D, W, M, attn::kBM, attn::kBN, (long long)dq_ctas,
      bs.dq_k_ring, bs.dq_v_ring, bs.dq_smem);
  if (t > 0 && n > 0 && n < (int)sizeof(out))
    n += snprintf(out + n, sizeof(out) - (size_t)n,
                  ",\"ttt_suffix\":{\"kernel\":\"ttt_diag_bwd_kernel<%d,%d>\","
                  "\"key_rows\":%lld}",
                  D, ch, (long long)p->B * p->Hkv * p->Sq);
  if (M && n > 0 && n < (int)sizeof(out))
    n += snprintf(out + n, sizeof(out) - (size_t)n,
                  ",\"mask_transpose\":{\"kernel\":\"mask_transpose_kernel\"}");
  if (n > 0 && n < (int)sizeof(out)) n += snprintf(out + n, sizeof(out) - (size_t)n, "}");
  if (n <= 0 || n >= (int)sizeof(out)) return fail(ATTN_ERR_INVALID, "description too long");
  if (needed != nullptr) *needed = (size_t)n + 1;
  if (buf == nullptr || buf_len < (size_t)n + 1)
    return fail(ATTN_ERR_INVALID, "describe: buffer of %zu bytes, %d needed", buf_len, n + 1);
  memcpy(buf, out, (size_t)n + 1);
  return ATTN_OK;
}

}  // extern "C"

namespace attn {

int fwd_split_tiles(const attn_problem* p) { return fwd_split_plan(make_dims(p)).split; }

size_t fwd_split_bytes(const attn_problem* p, int split) {
  return fwd_split_with(make_dims(p), split).bytes();
}

attn_status fwd_with_split(const attn_problem* p, int split, attn_tensor q, attn_tensor k,
                           attn_tensor v, attn_tensor o, float* lse, void* workspace,
                           size_t ws_bytes, void* stream) {
  attn_status st = check_problem(p);
  if (st != ATTN_OK) return st;
  if ((st = check_tensor(q, p->B, p->Hq, p->Sq, p->D, "q")) != ATTN_OK) return st;
  if ((st = check_tensor(k, p->B, p->Hkv, p->Skv, p->D, "k")) != ATTN_OK) return st;
  if ((st = check_tensor(v, p->B, p->Hkv, p->Skv, p->D, "v")) != ATTN_OK) return st;
  const int oes = p->out_dtype == ATTN_OUT_F32 ? 4 : 2;
  if ((st = check_tensor(o, p->B, p->Hq, p->Sq, p->D, "o", oes)) != ATTN_OK) return st;
  if (lse == nullptr) return fail(ATTN_ERR_INVALID, "lse is NULL");
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return fail(ATTN_ERR_ALIGNMENT, "lse is not 4-byte aligned");

  attn::FwdArgs a;
  a.d = make_dims(p);
  a.q = to_view(q);
  a.k = to_view(k);
  a.v = to_view(v);
  a.o = to_view(o);
  a.lse = lse;
  a.split = a.nchunk = 0;
  a.part_o = nullptr;
  a.part_ml = nullptr;
  const attn::FwdSplit sp = attn::fwd_split_with(a.d, split);
  if (sp.split > 0) {
    // the key range split over several CTAs (small grids): partials in the workspace
    if (workspace == nullptr) return fail(ATTN_ERR_WORKSPACE, "forward workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
      return fail(ATTN_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
    if (ws_bytes < sp.bytes())
      return fail(ATTN_ERR_WORKSPACE, "forward workspace too small: %zu < %zu bytes", ws_bytes,
                  sp.bytes());
    a.split = sp.split;
    a.nchunk = sp.nchunk;
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + sp.part_o_bytes);
  }
  if ((st = device_error_word(&a.ctl.err)) != ATTN_OK) return st;
  a.ctl.budget_ns = g_budget_ns.load();
  attn::Maps m;
  if ((st = make_map(&m.q, a.q, p->B, p->Hq, p->Sq, p->D, "q")) != ATTN_OK) return st;
  if ((st = make_map(&m.k, a.k, p->B, p->Hkv, p->Skv, p->D, "k")) != ATTN_OK) return st;
  if ((st = make_map(&m.v, a.v, p->B, p->Hkv, p->Skv, p->D, "v")) != ATTN_OK) return st;
  m.dout = m.q;
  NvtxRange range(a.split > 0 ? "attn_train_fwd:split" : "attn_train_fwd");
  cudaError_t e = attn::launch_fwd(a, m, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return ATTN_OK;
}

}  // namespace attn

extern "C" {

attn_status attn_train_bwd(const attn_problem* p, attn_tensor q, attn_tensor k, attn_tensor v,
                           attn_tensor o, attn_tensor dout, const float* lse, attn_tensor dq,
                           attn_tensor dk, attn_tensor dv, void* workspace, size_t ws_bytes,
                           void* stream) {
  return attn_train_bwd_passes(p, ATTN_BWD_ALL, q, k, v, o, dout, lse, dq, dk, dv, workspace,
                               ws_bytes, stream);
}

attn_status attn_train_bwd_passes(const attn_problem* p, unsigned passes, attn_tensor q,
                                  attn_tensor k, attn_tensor v, attn_tensor o, attn_tensor dout,
                                  const float* lse, attn_tensor dq, attn_tensor dk, attn_tensor dv,
                                  void* workspace, size_t ws_bytes, void* stream) {
  attn_status st = check_problem(p);
  if (st != ATTN_OK) return st;
  if (passes == 0 || (passes & ~(unsigned)ATTN_BWD_ALL) != 0)
    return fail(ATTN_ERR_INVALID, "passes mask 0x%x is empty or has unknown bits", passes);
  if ((st = check_tensor(q, p->B, p->Hq, p->Sq, p->D, "q")) != ATTN_OK) return st;
  if ((st = check_tensor(k, p->B, p->Hkv, p->Skv, p->D, "k")) != ATTN_OK) return st;
  if ((st = check_tensor(v, p->B, p->Hkv, p->Skv, p->D, "v")) != ATTN_OK) return st;
  const int oes = p->out_dtype == ATTN_OUT_F32 ? 4 : 2;
  if ((st = check_tensor(o, p->B, p->Hq, p->Sq, p->D, "o", oes)) != ATTN_OK) return st;
  if ((st = check_tensor(dout, p->B, p->Hq, p->Sq, p->D, "dout")) != ATTN_OK) return st;
  if ((st = check_tensor(dq, p->B, p->Hq, p->Sq, p->D, "dq", oes)) != ATTN_OK) return st;
  if ((st = check_tensor(dk, p->B, p->Hkv, p->Skv, p->D, "dk", oes)) != ATTN_OK) return st;
  if ((st = check_tensor(dv, p->B, p->Hkv, p->Skv, p->D, "dv", oes)) != ATTN_OK) return st;
  if (lse == nullptr) return fail(ATTN_ERR_INVALID, "lse is NULL");
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return fail(ATTN_ERR_ALIGNMENT, "lse is not 4-byte aligned");
  if (workspace == nullptr) return fail(ATTN_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
    return fail(ATTN_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
  if (ws_bytes < ws_bytes_for(p))
    return fail(ATTN_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes,
                ws_bytes_for(p));

  attn::BwdArgs a;
  a.d = make_dims(p);
  a.q = to_view(q);
  a.k = to_view(k);
  a.v = to_view(v);
  a.o = to_view(o);
  a.dout = to_view(dout);
  a.dq = to_view(dq);
  a.dk = to_view(dk);
  a.dv = to_view(dv);
  a.lse = lse;
  a.delta = static_cast<float*>(workspace);
  a.ttt_p = nullptr;
  a.ttt_ds = nullptr;
  if (ws_diag_bytes(p) > 0) {
    char* w = static_cast<char*>(workspace) + ws_delta_bytes(p);
    a.ttt_p = reinterpret_cast<float*>(w);
    a.ttt_ds = reinterpret_cast<float*>(w + ws_diag_bytes(p));
  }
  a.addm_t = nullptr;
  a.addm_t_sb = a.addm_t_sq = 0;
  if (p->add_mask != nullptr) {
    char* w = static_cast<char*>(workspace) + ws_delta_bytes(p) + 2 * ws_diag_bytes(p);
    a.addm_t = reinterpret_cast<uint16_t*>(w);
    a.addm_t_sq = mask_t_sq(p);
    a.addm_t_sb = p->add_mask_sb == 0 ? 0 : (int64_t)p->Skv * a.addm_t_sq;
  }
  if ((st = device_error_word(&a.ctl.err)) != ATTN_OK) return st;
  a.ctl.budget_ns = g_budget_ns.load();
  attn::Maps m;
  if ((st = make_map(&m.q, a.q, p->B, p->Hq, p->Sq, p->D, "q")) != ATTN_OK) return st;
  if ((st = make_map(&m.k, a.k, p->B, p->Hkv, p->Skv, p->D, "k")) != ATTN_OK) return st;
  if ((st = make_map(&m.v, a.v, p->B, p->Hkv, p->Skv, p->D, "v")) != ATTN_OK) return st;
  if ((st = make_map(&m.dout, a.dout, p->B, p->Hq, p->Sq, p->D, "dout")) != ATTN_OK) return st;
  cudaError_t e = cudaSuccess;
  if (nvtx_on()) {
    // one range per pass, launched one at a time in the usual order
    static const char* const names[4] = {"attn_train_bwd:prep", "attn_train_bwd:dkdv",
                                         "attn_train_bwd:dq", "attn_train_bwd:ttt_suffix"};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) {
      if ((passes & (1u << i)) == 0) continue;
      NvtxRange range(names[i]);
      e = attn::launch_bwd(a, m, 1u << i, static_cast<cudaStream_t>(stream));
    }
  } else {
    e = attn::launch_bwd(a, m, passes, static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return ATTN_OK;
}

attn_status attn_train_bwd_noalloc(const attn_problem* p, attn_tensor q, attn_tensor k,
                                   attn_tensor v, attn_tensor o, attn_tensor dout,
                                   const float* lse, attn_tensor dq, attn_tensor dk,
                                   attn_tensor dv, void* stream) {
  size_t need = 0;
  attn_status st = attn_train_workspace_size(p, &need);
  if (st != ATTN_OK) return st;
  if (need > kNoAllocScratchBytes)
    return fail(ATTN_ERR_WORKSPACE,
                "attn_train_bwd_noalloc: this problem's backward workspace is %zu bytes but the "
                "built-in scratch holds %zu bytes; call attn_train_bwd with a caller-provided "
                "workspace instead",
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != ATTN_OK) return st;
  return attn_train_bwd(p, q, k, v, o, dout, lse, dq, dk, dv, scratch, kNoAllocScratchBytes,
                        stream);
}

namespace {
attn_status check_loss_args(int64_t rows, int64_t V, const void* logits, int64_t ld_logits,
                            const void* target, int64_t ld_target, const void* mask) {
  if (rows <= 0 || V <= 0) return fail(ATTN_ERR_INVALID, "rows (%lld) and V (%lld) must be positive",
                                       (long long)rows, (long long)V);
  if (rows > 0x7fffffffLL || V > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "rows and V must fit in 31 bits");
  if (logits == nullptr || target == nullptr)
    return fail(ATTN_ERR_INVALID, "logits and target must not be NULL");
  if (ld_logits < V || ld_target < V)
    return fail(ATTN_ERR_INVALID, "row strides must be >= V");
  if (reinterpret_cast<uintptr_t>(logits) % 4 != 0 || reinterpret_cast<uintptr_t>(target) % 4 != 0)
    return fail(ATTN_ERR_ALIGNMENT, "logits and target must be 4-byte aligned");
  if (reinterpret_cast<uintptr_t>(mask) % 4 != 0)
    return fail(ATTN_ERR_ALIGNMENT, "mask must be 4-byte aligned");
  return ATTN_OK;
}
bool aligned4(const void* p) { return reinterpret_cast<uintptr_t>(p) % 4 == 0; }
}  // namespace

attn_status attn_train_logsoftmax_loss_fwd(int64_t rows, int64_t V, const float* logits,
                                           int64_t ld_logits, const float* target,
                                           int64_t ld_target, const float* mask,
                                           float* row_loss, float* row_lse, float* row_tsum,
                                           float* loss, void* stream) {
  attn_status st = check_loss_args(rows, V, logits, ld_logits, target, ld_target, mask);
  if (st != ATTN_OK) return st;
  if (row_loss == nullptr || row_lse == nullptr || row_tsum == nullptr)
    return fail(ATTN_ERR_INVALID, "row_loss, row_lse and row_tsum must not be NULL");
  if (!aligned4(row_loss) || !aligned4(row_lse) || !aligned4(row_tsum) || !aligned4(loss))
    return fail(ATTN_ERR_ALIGNMENT, "row outputs and loss must be 4-byte aligned");
  attn::LossArgs a{rows, V, ld_logits, ld_target, logits, nullptr, target, mask,
                   row_loss, row_lse, row_tsum, loss, nullptr};
  NvtxRange range("attn_train_logsoftmax_loss_fwd");
  cudaError_t e = attn::launch_logsoftmax_loss_fwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "log-softmax loss forward launch");
  return ATTN_OK;
}

attn_status attn_train_logsoftmax_loss_bwd(int64_t rows, int64_t V, float* logits,
                                           int64_t ld_logits, const float* target,
                                           int64_t ld_target, const float* mask,
                                           const float* row_lse, const float* row_tsum,
                                           const float* grad_loss, void* stream) {
  attn_status st = check_loss_args(rows, V, logits, ld_logits, target, ld_target, mask);
  if (st != ATTN_OK) return st;
  if (row_lse == nullptr || row_tsum == nullptr)
    return fail(ATTN_ERR_INVALID, "row_lse and row_tsum must not be NULL");
  if (!aligned4(row_lse) || !aligned4(row_tsum) || !aligned4(grad_loss))
    return fail(ATTN_ERR_ALIGNMENT, "row statistics and grad_loss must be 4-byte aligned");
  attn::LossArgs a{rows, V, ld_logits, ld_target, logits, logits, target, mask,
                   nullptr, const_cast<float*>(row_lse), const_cast<float*>(row_tsum), nullptr,
                   grad_loss};
  NvtxRange range("attn_train_logsoftmax_loss_bwd");
  cudaError_t e = attn::launch_logsoftmax_loss_bwd(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "log-softmax loss backward launch");
  return ATTN_OK;
}

const char* attn_train_last_error(void) { return g_msg; }

attn_status attn_train_device_status(void* stream) {
  uint32_t* w = nullptr;
  attn_status st = device_error_word(&w);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, w, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (word != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    if ((word & 0xffu) == attn::kErrDebugCheck)
      return fail(ATTN_ERR_DEVICE_CHECK, "a device-side check of the ATTN_DEBUG build failed "
                  "at site %u", word >> 8);
    return fail(ATTN_ERR_DEVICE_TIMEOUT, "a device-side wait ran out of budget (code %u)", word);
  }
  return ATTN_OK;
}

attn_status attn_train_set_wait_budget_ns(uint64_t ns) {
  g_budget_ns.store(ns < 1000000ull ? 1000000ull : ns);
  return ATTN_OK;
}

attn_status attn_train_mask_pattern(const attn_problem* p, uint8_t* bits, uint8_t* tiles,
                                    void* stream) {
  attn_status st = check_problem(p);
  if (st != ATTN_OK) return st;
  if (bits == nullptr) return fail(ATTN_ERR_INVALID, "bits is NULL");
  cudaError_t e = attn::launch_mask_pattern(make_dims(p), bits, tiles, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mask pattern launch");
  return ATTN_OK;
}

attn_status attn_train_probe_mma(int mode, int D, const void* a, const void* b, float* c,
                                 void* stream) {
  if (mode != 0 && mode != 1) return fail(ATTN_ERR_INVALID, "probe mode %d", mode);
  if (D != 16 && D != 32 && D != 64 && D != 128) return fail(ATTN_ERR_UNSUPPORTED, "probe D %d", D);
  if (a == nullptr || b == nullptr || c == nullptr) return fail(ATTN_ERR_INVALID, "probe NULL");
  if (reinterpret_cast<uintptr_t>(a) % 16 || reinterpret_cast<uintptr_t>(b) % 16)
    return fail(ATTN_ERR_ALIGNMENT, "probe operands not 16-byte aligned");
  Ctl ctl;
  attn_status st = device_error_word(&ctl.err);
  if (st != ATTN_OK) return st;
  ctl.budget_ns = g_budget_ns.load();
  View va{const_cast<void*>(a), 0, 0, mode == 0 ? D : 128};
  View vb{const_cast<void*>(b), 0, 0, D};
  CUtensorMap ta, tb;
  // mode 1 reads `a` with plain loads; its map is built but unused
  if ((st = make_map(&ta, va, 1, 1, 128, D, "probe a")) != ATTN_OK) return st;
  if ((st = make_map(&tb, vb, 1, 1, 128, D, "probe b")) != ATTN_OK) return st;
  cudaError_t e = attn::launch_probe(mode, D, ta, tb, a, c, ctl, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "probe launch");
  return ATTN_OK;
}

attn_status attn_train_selftest_debug_check(void* stream) {
  if (!attn::debug_checks_built())
    return fail(ATTN_ERR_UNSUPPORTED, "this library was built without ATTN_DEBUG");
  Ctl ctl;
  attn_status st = device_error_word(&ctl.err);
  if (st != ATTN_OK) return st;
  ctl.budget_ns = g_budget_ns.load();
  cudaError_t e = attn::launch_selftest_check(ctl, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return ATTN_OK;
}

attn_status attn_train_selftest_wait_timeout(void* stream) {
  Ctl ctl;
  attn_status st = device_error_word(&ctl.err);
  if (st != ATTN_OK) return st;
  ctl.budget_ns = 50000000ull;  // 50 ms
  cudaError_t e = attn::launch_selftest_wait(ctl, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return ATTN_OK;
}

}  // extern "C"
