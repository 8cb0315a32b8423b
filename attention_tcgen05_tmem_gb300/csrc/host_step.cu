// host_step.cu -- attn_train_step_host: one training step (forward and
// backward) whose inputs and outputs live in host memory.
//
// A step is one chunk (the whole problem), or chunks of whole GQA groups of
// one batch entry: kv head g of batch entry b, together with its query heads
// g*G .. g*G + G - 1, is an independent problem, and in the dense [B, H, S, D]
// host layout a run of such groups is one contiguous slice of every tensor.
// Three streams overlap the chunks:
//   copy-in   q, k, v, then dO of chunk c + 1 (while chunk c computes)
//   compute   forward; backward prep + dQ; backward dK/dV (the caller's stream)
//   copy-out  O and LSE during the backward, dQ during dK/dV, then dK, dV
// The device copies of a chunk live in one of n arena slots (n = 2 by
// default); chunk c + n takes chunk c's slot once chunk c's compute has read
// its inputs and its copy-out has read its outputs, so the copies may run up
// to n - 1 chunks ahead of (inputs) or behind (outputs) the kernels.  A
// session keeps the streams, events and slot counter between steps, so the
// chunks of the next step continue the rotation and its copy-in overlaps this
// step's compute.  Every chunk runs the same kernels as the device-memory
// entry points on the sub-problem, and no kernel mixes heads, so the results
// equal those of the unchunked call bit for bit.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <new>

#include "abi_internal.h"
#include "attn_train.h"
#include "kernels.h"

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxSlots = ATTN_HOST_MAX_SLOTS;
size_t up(size_t n) { return (n + kAlign - 1) & ~(kAlign - 1); }
int cdiv(int a, int b) { return (a + b - 1) / b; }

attn_status err(attn_status st, const char* msg) {
  return static_cast<attn_status>(attn::set_last_error(st, msg));
}

attn_status cuda_err(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  return err(ATTN_ERR_CUDA, buf);
}

// Chunks: kv_heads_per_chunk <= 0 makes the whole step one chunk (B batch
// entries); otherwise a chunk is up to that many kv heads of one batch entry.
// Within one step, smaller chunks shorten the copies that cannot overlap (the
// first chunk's inputs, the last chunk's dK and dV); across the steps of a
// session the copies overlap the neighbouring steps anyway, and smaller chunks
// only leave SMs idle at the end of every pass.
struct Plan {
  bool whole = true;  // one chunk of all B batch entries
  int NB = 0;         // batch entries per chunk (B when whole, else 1)
  int U = 0, per_b = 0, chunks = 0, G = 0, oes = 0;
  // offsets inside one slot and its size
  size_t s_q = 0, s_k = 0, s_v = 0, s_do = 0, s_o = 0, s_lse = 0, s_dq = 0, s_dk = 0, s_dv = 0;
  size_t slot = 0;
  int nslots = 2;  // chunk slots (and copies of the key lengths / mask)
  int fsplit = 0;  // the whole problem's forward split (chunk length in key tiles)
  // arena: static[nslots] (key lengths, mask) | chunk workspace | slot[nslots]
  size_t lens_off = 0, mask_off = 0, mask_bytes = 0, stat = 0, ws_off = 0, ws = 0, slot_off = 0;
  size_t total = 0;
};

// The sub-problem of nb batch entries with n kv heads each (device pointers
// for the key lengths and the mask, null when the problem has none).
attn_problem chunk_problem(const attn_problem& p, int nb, int n, const int32_t* lens,
                           const void* mask) {
  attn_problem s = p;
  s.B = nb;
  s.Hq = n * (p.Hq / p.Hkv);
  s.Hkv = n;
  s.seq_lengths = lens;
  s.add_mask = mask;
  return s;
}

attn_status make_plan(const attn_problem* p, int kv_heads_per_chunk, int slots, Plan* pl) {
  if (p == nullptr) return err(ATTN_ERR_INVALID, "problem is NULL");
  if (slots < 2 || slots > kMaxSlots)
    return err(ATTN_ERR_INVALID, "slots must be in [2, ATTN_HOST_MAX_SLOTS]");
  // Validate the problem as it will run on the device: the key lengths and the
  // mask are copied to 256-byte aligned arena offsets, so their host addresses
  // need no alignment; a stand-in aligned address takes their place for the
  // check (it is never dereferenced).
  attn_problem dp = *p;
  const void* aligned_stand_in = reinterpret_cast<const void*>(kAlign);
  if (p->seq_lengths != nullptr) dp.seq_lengths = static_cast<const int32_t*>(aligned_stand_in);
  if (p->add_mask != nullptr) dp.add_mask = aligned_stand_in;
  attn_status st = attn_train_supports(&dp);
  if (st != ATTN_OK) return st;
  if (kv_heads_per_chunk > p->Hkv)
    return err(ATTN_ERR_INVALID, "kv_heads_per_chunk exceeds Hkv");

  Plan& P = *pl;
  P.nslots = slots;
  P.whole = kv_heads_per_chunk <= 0;
  P.NB = P.whole ? p->B : 1;
  P.U = P.whole ? p->Hkv : kv_heads_per_chunk;
  P.per_b = cdiv(p->Hkv, P.U);
  P.chunks = P.whole ? 1 : p->B * P.per_b;
  P.G = p->Hq / p->Hkv;
  P.oes = p->out_dtype == ATTN_OUT_F32 ? 4 : 2;

  // elements of the q-shaped and k-shaped tensors of the largest chunk
  const size_t nq = (size_t)P.NB * P.U * P.G * p->Sq * p->D;
  const size_t nk = (size_t)P.NB * P.U * p->Skv * p->D;
  size_t o = 0;
  P.s_q = o;   o += up(nq * 2);
  P.s_k = o;   o += up(nk * 2);
  P.s_v = o;   o += up(nk * 2);
  P.s_do = o;  o += up(nq * 2);
  P.s_o = o;   o += up(nq * P.oes);
  P.s_lse = o; o += up((size_t)P.NB * P.U * P.G * p->Sq * 4);
  P.s_dq = o;  o += up(nq * P.oes);
  P.s_dk = o;  o += up(nk * P.oes);
  P.s_dv = o;  o += up(nk * P.oes);
  P.slot = o;

  o = 0;
  P.lens_off = o;
  if (p->seq_lengths != nullptr) o += up((size_t)p->B * 4);
  P.mask_off = o;
  if (p->add_mask != nullptr) {
    const int64_t Bm = p->add_mask_sb == 0 ? 1 : p->B;
    P.mask_bytes = (size_t)((Bm - 1) * p->add_mask_sb + (int64_t)(p->Sq - 1) * p->add_mask_sq +
                            p->Skv) * 2;
    o += up(P.mask_bytes);
  }
  P.stat = o;
  o = (size_t)slots * P.stat;
  // one workspace region serves the forward's key-range split and the backward:
  // the forward's merge pass has consumed its partials before the backward runs.
  // Every chunk splits its forward like the whole problem would, so that the
  // chunked results equal the whole problem's bit for bit.
  attn_problem cp = chunk_problem(dp, P.NB, P.U, dp.seq_lengths, dp.add_mask);
  if ((st = attn_train_workspace_size(&cp, &P.ws)) != ATTN_OK) return st;
  P.fsplit = attn::fwd_split_tiles(&dp);
  const size_t fws = attn::fwd_split_bytes(&cp, P.fsplit);
  if (fws > P.ws) P.ws = fws;
  P.ws_off = o;
  o += up(P.ws);
  P.slot_off = o;
  o += (size_t)slots * P.slot;
  P.total = o;
  return ATTN_OK;
}

attn_tensor dev_view(const void* ptr, int H, int S, int D) {
  attn_tensor t;
  t.ptr = ptr;
  t.stride_b = (int64_t)H * S * D;  // dense [nb, H, S, D]
  t.stride_h = (int64_t)S * D;
  t.stride_s = D;
  return t;
}

}  // namespace

// A session: the problem, its plan and arena, the two copy streams and the
// events that order the slots.  Chunks take the slots in turn across steps,
// so the next step's copy-in overlaps this step's compute.
struct attn_host_session_s {
  attn_problem p{};
  Plan pl;
  char* arena = nullptr;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, stat = nullptr, end_in = nullptr, end_out = nullptr;
  // per slot (only the first pl.nslots exist): compute of the last step that
  // used static area i; per chunk slot: its inputs copied (q, k, v / all),
  // its forward, its dQ pass and its whole backward computed, its outputs copied
  cudaEvent_t step_done[kMaxSlots] = {};
  cudaEvent_t qkv[kMaxSlots] = {}, inp[kMaxSlots] = {}, fwd[kMaxSlots] = {},
              dq[kMaxSlots] = {}, bwd[kMaxSlots] = {}, outd[kMaxSlots] = {};
  int64_t chunk = 0;    // chunks enqueued so far (slot = chunk % nslots)
  int64_t step = 0;     // steps enqueued so far (static area = step % nslots)
  bool failed = false;  // a step stopped part-way: the slot bookkeeping no longer
                        // matches what was enqueued, so no further step is accepted

  template <typename F>
  void each_event(F f) {
    f(&start);
    f(&stat);
    f(&end_in);
    f(&end_out);
    for (int i = 0; i < pl.nslots; ++i) {
      f(&step_done[i]);
      f(&qkv[i]);
      f(&inp[i]);
      f(&fwd[i]);
      f(&dq[i]);
      f(&bwd[i]);
      f(&outd[i]);
    }
  }
  cudaError_t create() {
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    e = cudaSuccess;
    each_event([&](cudaEvent_t* ev) {
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    });
    return e;
  }
  // A stream or event destroyed with work pending is released once that work completes.
  ~attn_host_session_s() {
    each_event([](cudaEvent_t* ev) {
      if (*ev != nullptr) cudaEventDestroy(*ev);
    });
    if (in != nullptr) cudaStreamDestroy(in);
    if (out != nullptr) cudaStreamDestroy(out);
  }

  attn_status enqueue_step(const attn_host_io* io, cudaStream_t cs);
  attn_status join(cudaStream_t cs);
};

attn_status attn_host_session_s::enqueue_step(const attn_host_io* io, cudaStream_t cs) {
  const attn_problem& P = p;
  const auto H2D = cudaMemcpyHostToDevice;
  const auto D2H = cudaMemcpyDeviceToHost;
  const char* hq = static_cast<const char*>(io->q);
  const char* hk = static_cast<const char*>(io->k);
  const char* hv = static_cast<const char*>(io->v);
  const char* hdo = static_cast<const char*>(io->dout);
  char* ho = static_cast<char*>(io->o);
  char* hlse = reinterpret_cast<char*>(io->lse);
  char* hdq = static_cast<char*>(io->dq);
  char* hdk = static_cast<char*>(io->dk);
  char* hdv = static_cast<char*>(io->dv);
  cudaError_t e = cudaSuccess;
  attn_status st = ATTN_OK;
#define STEP_CUDA(call, name)       \
  do {                              \
    if ((e = (call)) != cudaSuccess) \
      return cuda_err(e, (name));   \
  } while (0)

  if (step == 0) {
    // the arena may still be in use by work enqueued on `stream` before the session
    STEP_CUDA(cudaEventRecord(start, cs), "event record");
    STEP_CUDA(cudaStreamWaitEvent(in, start, 0), "stream wait");
    STEP_CUDA(cudaStreamWaitEvent(out, start, 0), "stream wait");
  }
  // every step shares the chunk workspace: compute follows the previous step's
  // compute even when the caller passes another stream
  const int ns = pl.nslots;
  const int par = (int)(step % ns);
  if (step >= 1)
    STEP_CUDA(cudaStreamWaitEvent(cs, step_done[(step - 1) % ns], 0), "stream wait");
  // key lengths and mask: static area step % n, free once step - n has been computed
  char* stat_area = arena + (size_t)par * pl.stat;
  if (step >= ns) STEP_CUDA(cudaStreamWaitEvent(in, step_done[par], 0), "stream wait");
  if (P.seq_lengths != nullptr)
    STEP_CUDA(cudaMemcpyAsync(stat_area + pl.lens_off, P.seq_lengths, (size_t)P.B * 4, H2D, in),
              "key lengths copy-in");
  if (P.add_mask != nullptr)
    STEP_CUDA(cudaMemcpyAsync(stat_area + pl.mask_off, P.add_mask, pl.mask_bytes, H2D, in),
              "mask copy-in");
  STEP_CUDA(cudaEventRecord(stat, in), "event record");
  STEP_CUDA(cudaStreamWaitEvent(cs, stat, 0), "stream wait");

  for (int b = 0; b < P.B; b += pl.NB) {
    for (int j = 0; j < pl.per_b; ++j, ++chunk) {
      // this chunk: batch entries [b, b + NB), kv heads [g0, g0 + n)
      const int g0 = j * pl.U;
      const int n = (P.Hkv - g0) < pl.U ? (P.Hkv - g0) : pl.U;
      const int hq_n = n * pl.G;
      const int nb = pl.NB;
      const int s = (int)(chunk % ns);
      char* S = arena + pl.slot_off + (size_t)s * pl.slot;
      const int32_t* lens =
          P.seq_lengths ? reinterpret_cast<const int32_t*>(stat_area + pl.lens_off) + b : nullptr;
      const void* mask =
          P.add_mask
              ? stat_area + pl.mask_off + (size_t)(P.add_mask_sb == 0 ? 0 : b * P.add_mask_sb) * 2
              : nullptr;
      const attn_problem sp = chunk_problem(P, nb, n, lens, mask);
      // host element offsets and counts of this chunk's slices (contiguous: a chunk
      // is either part of one batch entry's heads or whole batch entries)
      const size_t eq = ((size_t)b * P.Hq + (size_t)g0 * pl.G) * P.Sq * P.D;
      const size_t ek = ((size_t)b * P.Hkv + g0) * P.Skv * P.D;
      const size_t el = ((size_t)b * P.Hq + (size_t)g0 * pl.G) * P.Sq;
      const size_t nq = (size_t)nb * hq_n * P.Sq * P.D, nk = (size_t)nb * n * P.Skv * P.D;
      const size_t nl = (size_t)nb * hq_n * P.Sq;

      // copy-in: the slot's inputs are free once chunk - n has been computed
      if (chunk >= ns) STEP_CUDA(cudaStreamWaitEvent(in, bwd[s], 0), "stream wait");
      STEP_CUDA(cudaMemcpyAsync(S + pl.s_q, hq + eq * 2, nq * 2, H2D, in), "q copy-in");
      STEP_CUDA(cudaMemcpyAsync(S + pl.s_k, hk + ek * 2, nk * 2, H2D, in), "k copy-in");
      STEP_CUDA(cudaMemcpyAsync(S + pl.s_v, hv + ek * 2, nk * 2, H2D, in), "v copy-in");
      STEP_CUDA(cudaEventRecord(qkv[s], in), "event record");
      STEP_CUDA(cudaMemcpyAsync(S + pl.s_do, hdo + eq * 2, nq * 2, H2D, in), "dout copy-in");
      STEP_CUDA(cudaEventRecord(inp[s], in), "event record");

      // compute: the slot's outputs are free once chunk - n has been copied out
      const attn_tensor q = dev_view(S + pl.s_q, hq_n, P.Sq, P.D);
      const attn_tensor k = dev_view(S + pl.s_k, n, P.Skv, P.D);
      const attn_tensor v = dev_view(S + pl.s_v, n, P.Skv, P.D);
      const attn_tensor dout = dev_view(S + pl.s_do, hq_n, P.Sq, P.D);
      const attn_tensor o = dev_view(S + pl.s_o, hq_n, P.Sq, P.D);
      const attn_tensor dqv = dev_view(S + pl.s_dq, hq_n, P.Sq, P.D);
      const attn_tensor dk = dev_view(S + pl.s_dk, n, P.Skv, P.D);
      const attn_tensor dv = dev_view(S + pl.s_dv, n, P.Skv, P.D);
      float* lse = reinterpret_cast<float*>(S + pl.s_lse);
      void* ws = arena + pl.ws_off;
      STEP_CUDA(cudaStreamWaitEvent(cs, qkv[s], 0), "stream wait");
      if (chunk >= ns) STEP_CUDA(cudaStreamWaitEvent(cs, outd[s], 0), "stream wait");
      if ((st = attn::fwd_with_split(&sp, pl.fsplit, q, k, v, o, lse, ws, pl.ws, cs)) != ATTN_OK)
        return st;
      STEP_CUDA(cudaEventRecord(fwd[s], cs), "event record");
      STEP_CUDA(cudaStreamWaitEvent(cs, inp[s], 0), "stream wait");
      if ((st = attn_train_bwd_passes(&sp, ATTN_BWD_PREP | ATTN_BWD_DQ, q, k, v, o, dout, lse, dqv,
                                      dk, dv, ws, pl.ws, cs)) != ATTN_OK)
        return st;
      STEP_CUDA(cudaEventRecord(dq[s], cs), "event record");
      if ((st = attn_train_bwd_passes(&sp, ATTN_BWD_DKDV | ATTN_BWD_TTT, q, k, v, o, dout, lse,
                                      dqv, dk, dv, ws, pl.ws, cs)) != ATTN_OK)
        return st;
      STEP_CUDA(cudaEventRecord(bwd[s], cs), "event record");

      // copy-out
      STEP_CUDA(cudaStreamWaitEvent(out, fwd[s], 0), "stream wait");
      STEP_CUDA(cudaMemcpyAsync(ho + eq * pl.oes, S + pl.s_o, nq * pl.oes, D2H, out),
                "o copy-out");
      STEP_CUDA(cudaMemcpyAsync(hlse + el * 4, S + pl.s_lse, nl * 4, D2H, out), "lse copy-out");
      STEP_CUDA(cudaStreamWaitEvent(out, dq[s], 0), "stream wait");
      STEP_CUDA(cudaMemcpyAsync(hdq + eq * pl.oes, S + pl.s_dq, nq * pl.oes, D2H, out),
                "dq copy-out");
      STEP_CUDA(cudaStreamWaitEvent(out, bwd[s], 0), "stream wait");
      STEP_CUDA(cudaMemcpyAsync(hdk + ek * pl.oes, S + pl.s_dk, nk * pl.oes, D2H, out),
                "dk copy-out");
      STEP_CUDA(cudaMemcpyAsync(hdv + ek * pl.oes, S + pl.s_dv, nk * pl.oes, D2H, out),
                "dv copy-out");
      STEP_CUDA(cudaEventRecord(outd[s], out), "event record");
    }
  }
  STEP_CUDA(cudaEventRecord(step_done[par], cs), "event record");
  ++step;
#undef STEP_CUDA
  return ATTN_OK;
}

attn_status attn_host_session_s::join(cudaStream_t cs) {
  cudaError_t e = cudaEventRecord(end_in, in);
  if (e == cudaSuccess) e = cudaEventRecord(end_out, out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, end_in, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, end_out, 0);
  return e == cudaSuccess ? ATTN_OK : cuda_err(e, "joining the copy streams");
}

namespace {

attn_status check_io(const attn_host_io* io) {
  if (io == nullptr) return err(ATTN_ERR_INVALID, "io is NULL");
  if (io->q == nullptr || io->k == nullptr || io->v == nullptr || io->dout == nullptr ||
      io->o == nullptr || io->lse == nullptr || io->dq == nullptr || io->dk == nullptr ||
      io->dv == nullptr)
    return err(ATTN_ERR_INVALID, "a host buffer of io is NULL");
  return ATTN_OK;
}

attn_status check_arena(const Plan& pl, void* arena, size_t arena_bytes) {
  if (arena == nullptr) return err(ATTN_ERR_WORKSPACE, "arena is NULL");
  if (reinterpret_cast<uintptr_t>(arena) % kAlign != 0)
    return err(ATTN_ERR_ALIGNMENT, "arena is not 256-byte aligned");
  if (arena_bytes < pl.total) {
    char buf[160];
    snprintf(buf, sizeof(buf), "arena too small: %zu < %zu bytes", arena_bytes, pl.total);
    return err(ATTN_ERR_WORKSPACE, buf);
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_train_host_session_arena_size(const attn_problem* p, int kv_heads_per_chunk,
                                               int slots, size_t* bytes) {
  Plan pl;
  attn_status st = make_plan(p, kv_heads_per_chunk, slots, &pl);
  if (st != ATTN_OK) return st;
  if (bytes == nullptr) return err(ATTN_ERR_INVALID, "bytes is NULL");
  *bytes = pl.total;
  return ATTN_OK;
}

attn_status attn_train_step_host_arena_size(const attn_problem* p, int kv_heads_per_chunk,
                                            size_t* bytes) {
  return attn_train_host_session_arena_size(p, kv_heads_per_chunk, 2, bytes);
}

attn_status attn_train_host_session_create_slots(const attn_problem* p, int kv_heads_per_chunk,
                                                 int slots, void* arena, size_t arena_bytes,
                                                 attn_host_session* out) {
  if (out == nullptr) return err(ATTN_ERR_INVALID, "out is NULL");
  *out = nullptr;
  Plan pl;
  attn_status st = make_plan(p, kv_heads_per_chunk, slots, &pl);
  if (st != ATTN_OK) return st;
  if ((st = check_arena(pl, arena, arena_bytes)) != ATTN_OK) return st;
  attn_host_session_s* s = new (std::nothrow) attn_host_session_s();
  if (s == nullptr) return err(ATTN_ERR_INVALID, "out of host memory");
  s->p = *p;
  s->pl = pl;
  s->arena = static_cast<char*>(arena);
  cudaError_t e = s->create();
  if (e != cudaSuccess) {
    delete s;
    return cuda_err(e, "stream/event creation");
  }
  *out = s;
  return ATTN_OK;
}

attn_status attn_train_host_session_create(const attn_problem* p, int kv_heads_per_chunk,
                                           void* arena, size_t arena_bytes,
                                           attn_host_session* out) {
  return attn_train_host_session_create_slots(p, kv_heads_per_chunk, 2, arena, arena_bytes, out);
}

attn_status attn_train_host_session_step(attn_host_session s, const attn_host_io* io,
                                         void* stream) {
  if (s == nullptr) return err(ATTN_ERR_INVALID, "session is NULL");
  if (s->failed)
    return err(ATTN_ERR_INVALID,
               "an earlier step of this session failed part-way; join, synchronize and "
               "destroy it, then create a new session");
  attn_status st = check_io(io);
  if (st != ATTN_OK) return st;
  st = s->enqueue_step(io, static_cast<cudaStream_t>(stream));
  if (st != ATTN_OK) s->failed = true;
  return st;
}

attn_status attn_train_host_session_join(attn_host_session s, void* stream) {
  if (s == nullptr) return err(ATTN_ERR_INVALID, "session is NULL");
  return s->join(static_cast<cudaStream_t>(stream));
}

attn_status attn_train_host_session_destroy(attn_host_session s) {
  delete s;
  return ATTN_OK;
}

attn_status attn_train_step_host(const attn_problem* p, const attn_host_io* io,
                                 int kv_heads_per_chunk, void* arena, size_t arena_bytes,
                                 void* stream) {
  attn_status st = check_io(io);
  if (st != ATTN_OK) {
    // report a malformed problem first, as the other entry points do
    Plan pl;
    attn_status pst = make_plan(p, kv_heads_per_chunk, 2, &pl);
    return pst != ATTN_OK ? pst : check_io(io);
  }
  attn_host_session s = nullptr;
  if ((st = attn_train_host_session_create(p, kv_heads_per_chunk, arena, arena_bytes, &s)) !=
      ATTN_OK)
    return st;
  st = s->enqueue_step(io, static_cast<cudaStream_t>(stream));
  // `stream` waits for every copy enqueued, also after a failure, so that no
  // copy outlives the caller's buffers unseen
  const attn_status jst = s->join(static_cast<cudaStream_t>(stream));
  delete s;
  return st != ATTN_OK ? st : jst;
}

}  // extern "C"
