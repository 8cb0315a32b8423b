// kernels.h -- internal interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; the public interface is
// include/attn_train.h.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sched.cuh"

namespace attn {

// A [B, H, S, D] bf16 view; strides in elements, D stride 1.
struct View {
  void* ptr;
  int64_t sb, sh, ss;
};

struct Dims {
  int B, Hq, Hkv, Sq, Skv, D, G;
  MaskGeom geom;
  float scale;       // softmax scale c
  float scale_log2;  // c * log2(e)
  int out_f32;       // O, dQ, dK, dV are fp32 (else bf16)
  const int* seqlens;  // device [B]: key length of each batch entry, or null (all keys)
  // additive mask (bf16 bits): element (b, q, kv) at addm[b * addm_sb + q * addm_sq + kv]
  const uint16_t* addm;
  int64_t addm_sb, addm_sq;
};

// Whether a problem needs the general mask arithmetic: a window mask (two-sided
// bounds), per-batch key lengths or an additive mask.
inline bool needs_general_mask(const Dims& d) {
  return d.geom.kind == kMaskWindow || d.seqlens != nullptr || d.addm != nullptr;
}

struct Ctl {
  uint32_t* err;       // device error word
  uint64_t budget_ns;  // per-wait budget
};

struct FwdArgs {
  Dims d;
  View q, k, v, o;
  float* lse;  // [B, Hq, Sq]
  Ctl ctl;
  // Split over key tiles (see FwdSplit): split = key tiles per chunk (0: one CTA
  // per query-tile pair, writing O and LSE itself); nchunk = chunk slots per pair;
  // part_o [B*Hq][n_qp][nchunk][2*kBM][D] and part_ml [same slots][2*kBM] (running
  // max and sum) in the workspace.
  int split, nchunk;
  float* part_o;
  float2* part_ml;
};

// The forward's key-range split for grids that would leave most SMs idle: each
// query-tile pair's key tiles are cut into chunks of `split` tiles, one CTA per
// (pair, chunk), and a merge pass combines the chunks' partial results in chunk
// order.  split = 0: no split.
struct FwdSplit {
  int split = 0, nchunk = 0;
  size_t part_o_bytes = 0, part_ml_bytes = 0;
  size_t bytes() const { return part_o_bytes + part_ml_bytes; }
};
// Planned for kPlanSMs multiprocessors (a GB300's count): the plan only changes
// scheduling, so it is a pure function of the problem (workspace sizes can be
// computed without a device, and a device with another count still gets exact
// results).
constexpr int kPlanSMs = 152;
FwdSplit fwd_split_plan(const Dims& d);
// The layout of a split into chunks of `split` key tiles for this problem (split
// <= 0 or a TTT mask: none); slices of a larger problem use the larger problem's
// chunk length, so that their results equal its results bit for bit.
FwdSplit fwd_split_with(const Dims& d, int split);

struct BwdArgs {
  Dims d;
  View q, k, v, o, dout, dq, dk, dv;
  const float* lse;  // [B, Hq, Sq]
  float* delta;      // workspace [B, Hq, Sq]
  // TTT only (else null): per query row, the weight p_i and the score
  // gradient ds_i of its suffix diagonal i = 1..t, workspace [B, Hq, Sq, t]
  float* ttt_p;
  float* ttt_ds;
  // additive mask transposed by the prep pass (workspace): element (b, kv, q) at
  // addm_t[b * addm_t_sb + kv * addm_t_sq + q]; null without an additive mask
  uint16_t* addm_t;
  int64_t addm_t_sb, addm_t_sq;
  Ctl ctl;
};

struct Maps {
  CUtensorMap q, k, v, dout;
};

// Soft-target log-softmax loss over [rows, V] fp32 logits (loss.cu).
struct LossArgs {
  int64_t rows, V, ld_logits, ld_target;  // row strides in elements
  const float* logits;                    // forward input
  float* logits_out;                      // backward: logits in, gradient out (in place)
  const float* target;
  const float* mask;       // [rows] or null (all ones)
  float* row_loss;         // [rows]: -sum_v target * log_softmax (before the mask)
  float* row_lse;          // [rows]: logsumexp of the row
  float* row_tsum;         // [rows]: sum_v target
  float* loss;             // [1] mean loss, or null (forward)
  const float* grad_loss;  // [1] upstream gradient, or null = 1 (backward)
};
cudaError_t launch_logsoftmax_loss_fwd(const LossArgs& a, cudaStream_t s);
cudaError_t launch_logsoftmax_loss_bwd(const LossArgs& a, cudaStream_t s);

// Pipeline shapes of the kernels a problem runs (attn_train_describe).
struct FwdShape {
  int ring = 0;                // K/V ring entries (128-key K or V tiles)
  bool three_buffers = false;  // three rotating score buffers (general masks, D <= 64)
  int smem = 0;                // dynamic shared memory per CTA, bytes
};
FwdShape fwd_shape(const Dims& d);
struct BwdShape {
  int dkdv_stages = 0, dq_k_ring = 0, dq_v_ring = 0, dkdv_smem = 0, dq_smem = 0;
};
BwdShape bwd_shape(int D);

cudaError_t launch_fwd(const FwdArgs& a, const Maps& m, cudaStream_t s);
// The split forward (a.split > 0) and its merge pass (fwd_split.cu).
cudaError_t launch_fwd_split(const FwdArgs& a, const Maps& m, cudaStream_t s);
// passes: mask of 1 = Delta prep, 2 = dK/dV, 4 = dQ, 8 = TTT suffix keys
cudaError_t launch_bwd(const BwdArgs& a, const Maps& m, unsigned passes, cudaStream_t s);
cudaError_t launch_mask_pattern(const Dims& d, uint8_t* bits, uint8_t* tiles, cudaStream_t s);
// One-tile descriptor probe (test only).  mode 0: C[128x128] = A[128xD] B[128xD]^T with
// both operands K-major in shared memory; mode 1: C[128xD] = A[128x128] B[128xD] with A in
// tensor memory and B MN-major in shared memory.
cudaError_t launch_probe(int mode, int D, const CUtensorMap& ta, const CUtensorMap& tb,
                         const void* a_global, float* c, Ctl ctl, cudaStream_t s);
cudaError_t launch_selftest_wait(Ctl ctl, cudaStream_t s);
// Whether this library was built with -DATTN_DEBUG (device-side checks), and a
// kernel whose check fails on purpose (only meaningful when it was).
bool debug_checks_built();
cudaError_t launch_selftest_check(Ctl ctl, cudaStream_t s);

// Records `msg` as the calling thread's last error message (attn_train_last_error)
// and returns `status`; for host code outside the C ABI's own translation unit.
int set_last_error(int status, const char* msg);

}  // namespace attn
