// step.cu -- one hybrid-batch step from host memory (hb_step and its slot
// objects), for a serving loop that keeps a few steps in flight.
//
// A step crosses the host link with one copy each way: the step's inputs
// (q, k_new, v_new and the batch descriptors) travel as one packed block
// (hb_step_layout), the output as one array.  The plan is built on the host
// and uploaded on the input-copy stream ahead of the inputs, the append and
// the attention run on the compute stream, the output comes back on the
// output-copy stream.  After its copies the input-copy stream writes the
// step's sequence number into a flag of the slot, and the append kernel
// polls that flag (bounded) before it reads its inputs and lets the attention
// kernel start: the compute stream carries no event wait between two steps,
// so each step's append still launches under the previous attention's tail
// (programmatic dependent launch needs the two kernels back to back on the
// stream; a wait between them measured 0.90 of the device rate end to end on
// a 106 us step).  The output copy is ordered by the slot's events, and the
// kernels wait for the slot's previous output copy only if it has not
// finished by the time the step is issued.  The kernels are those of
// hb_kv_append and hb_attention_new_kv (the chunks read their new K/V rows
// from the packed block rather than after the append).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <new>

#include "hb.h"

namespace hb {
hb_status internal_fail(hb_status s, const char* msg);   // message for hb_last_error
hb_status internal_ok();
hb_status internal_kv_append(const hb_batch* batch, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, void* stream,
                             const uint32_t* ready_flag, uint32_t ready_value);
}  // namespace hb

namespace {

constexpr size_t kStepAlign = 256;

size_t align_up(size_t x) { return (x + kStepAlign - 1) / kStepAlign * kStepAlign; }

hb_status step_fail(hb_status s, const char* msg) { return hb::internal_fail(s, msg); }

// cuStreamWriteValue32 from the driver (fetched once)
using WriteValue32 = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
WriteValue32 write_value32() {
  static std::once_flag once;
  static WriteValue32 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WriteValue32>(f);
  });
  return fn;
}

// Sizes of the packed input block's sections, in order: q, k_new, v_new,
// cu_q_len, context_len, block_table.
void section_bytes(const hb_batch* b, size_t out[HB_STEP_SECTIONS]) {
  const size_t T = (size_t)b->total_q, S = (size_t)b->num_seqs;
  out[0] = T * (size_t)b->num_q_heads * (size_t)b->head_dim * 2;
  out[1] = T * (size_t)b->num_kv_heads * (size_t)b->head_dim * 2;
  out[2] = out[1];
  out[3] = (S + 1) * 4;
  out[4] = S * 4;
  out[5] = S * (size_t)b->max_pages_per_seq * 4;
}

}  // namespace

struct hb_step_slot {
  int device = -1;
  cudaEvent_t in = nullptr;    // the step's inputs (and plan) are on the device
  cudaEvent_t done = nullptr;  // its kernels are done with them
  cudaEvent_t out = nullptr;   // its output has reached the host
  uint32_t* flag = nullptr;    // device word: sequence number of the last input copy
  uint32_t seq = 0;            // that of the last step issued on this slot
};

extern "C" {

hb_status hb_step_layout(const hb_batch* shape, size_t offsets[HB_STEP_SECTIONS],
                         size_t* in_bytes) {
  if (!shape || !offsets || !in_bytes) return step_fail(HB_ERR_INVALID_ARG, "NULL argument");
  if (shape->num_seqs < 0 || shape->total_q < 0 || shape->num_q_heads <= 0 ||
      shape->num_kv_heads <= 0 || shape->head_dim <= 0 || shape->max_pages_per_seq <= 0)
    return step_fail(HB_ERR_SHAPE, "sizes must be positive (num_seqs, total_q >= 0)");
  size_t n[HB_STEP_SECTIONS];
  section_bytes(shape, n);
  size_t off = 0;
  for (int i = 0; i < HB_STEP_SECTIONS; ++i) {
    offsets[i] = off;
    off = align_up(off + n[i]);
  }
  *in_bytes = off;
  return hb::internal_ok();
}

hb_status hb_step_slot_create(hb_step_slot** out) {
  if (!out) return step_fail(HB_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  hb_step_slot* s = new (std::nothrow) hb_step_slot;
  if (!s) return step_fail(HB_ERR_CUDA, "out of host memory");
  if (cudaGetDevice(&s->device) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->done, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->out, cudaEventDisableTiming) != cudaSuccess) {
    hb_step_slot_destroy(s);
    return step_fail(HB_ERR_CUDA, "creating the slot's events failed");
  }
  if (cudaMalloc(&s->flag, sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(s->flag, 0, sizeof(uint32_t)) != cudaSuccess) {
    hb_step_slot_destroy(s);
    return step_fail(HB_ERR_CUDA, "allocating the slot's flag failed");
  }
  if (!write_value32()) {
    hb_step_slot_destroy(s);
    return step_fail(HB_ERR_CUDA, "cuStreamWriteValue32 is not available");
  }
  *out = s;
  return hb::internal_ok();
}

void hb_step_slot_destroy(hb_step_slot* s) {
  if (!s) return;
  if (s->in) cudaEventDestroy(s->in);
  if (s->done) cudaEventDestroy(s->done);
  if (s->out) cudaEventDestroy(s->out);
  if (s->flag) cudaFree(s->flag);
  delete s;
}

hb_status hb_step_slot_sync(hb_step_slot* s) {
  if (!s) return step_fail(HB_ERR_INVALID_ARG, "NULL slot");
  if (cudaEventSynchronize(s->out) != cudaSuccess ||
      cudaEventSynchronize(s->done) != cudaSuccess ||
      cudaEventSynchronize(s->in) != cudaSuccess)
    return step_fail(HB_ERR_CUDA, "waiting for the slot's last step failed");
  return hb::internal_ok();
}

hb_status hb_step(const hb_batch* shape, const int32_t* h_q_len, const int32_t* h_context_len,
                  int32_t num_sms, hb_step_slot* slot, const hb_step_buffers* buf,
                  void* k_cache, void* v_cache, float softmax_scale, void* copy_in_stream,
                  void* stream, void* copy_out_stream) {
  try {
    if (!shape || !slot || !buf) return step_fail(HB_ERR_INVALID_ARG, "NULL argument");
    if (!buf->h_in || !buf->d_in || !buf->h_out || !buf->d_out || !buf->h_plan ||
        !buf->d_workspace)
      return step_fail(HB_ERR_INVALID_ARG, "every buffer of hb_step_buffers must be non-NULL");
    if ((reinterpret_cast<uintptr_t>(buf->d_in) & (kStepAlign - 1)) ||
        (reinterpret_cast<uintptr_t>(buf->d_out) & 15u))
      return step_fail(HB_ERR_INVALID_ARG,
                       "d_in must be 256-byte aligned and d_out 16-byte aligned");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != slot->device)
      return step_fail(HB_ERR_INVALID_ARG, "the slot belongs to another device");
    size_t off[HB_STEP_SECTIONS], in_bytes = 0;
    hb_status s = hb_step_layout(shape, off, &in_bytes);
    if (s != HB_OK) return s;
    if (shape->total_q == 0) return HB_OK;
    uint8_t* d_in = static_cast<uint8_t*>(buf->d_in);
    hb_batch b = *shape;
    b.cu_q_len = reinterpret_cast<const int32_t*>(d_in + off[3]);
    b.context_len = reinterpret_cast<const int32_t*>(d_in + off[4]);
    b.block_table = reinterpret_cast<const int32_t*>(d_in + off[5]);
    cudaStream_t s_in = static_cast<cudaStream_t>(copy_in_stream);
    cudaStream_t s_run = static_cast<cudaStream_t>(stream);
    cudaStream_t s_out = static_cast<cudaStream_t>(copy_out_stream);

    // the slot's last upload from h_plan has to be over before the plan is
    // rewritten (a page-locked plan is copied asynchronously); by the time a
    // slot comes round again it normally is
    if (cudaEventSynchronize(slot->in) != cudaSuccess)
      return step_fail(HB_ERR_CUDA, "waiting for the slot's last upload failed");
    // inputs: after the slot's last kernels are done with d_in and the
    // workspace, the plan (ahead of the bulk copy) and the packed block
    if (cudaStreamWaitEvent(s_in, slot->done, 0) != cudaSuccess)
      return step_fail(HB_ERR_CUDA, "ordering the input copy failed");
    size_t pb = buf->plan_bytes, wb = buf->workspace_bytes;
    s = hb_plan(&b, h_q_len, h_context_len, num_sms, buf->h_plan, &pb, buf->d_workspace, &wb,
                copy_in_stream);
    if (s != HB_OK) return s;
    if (cudaMemcpyAsync(d_in, buf->h_in, in_bytes, cudaMemcpyHostToDevice, s_in) != cudaSuccess)
      return step_fail(HB_ERR_CUDA, "the input copy failed");
    // then the flag: the copies before it on this stream are complete and
    // visible when the value lands
    const uint32_t seq = slot->seq + 1;
    if (write_value32()(reinterpret_cast<CUstream>(s_in), reinterpret_cast<CUdeviceptr>(slot->flag),
                        seq, 0) != CUDA_SUCCESS ||
        cudaEventRecord(slot->in, s_in) != cudaSuccess)
      return step_fail(HB_ERR_CUDA, "raising the slot's flag failed");
    slot->seq = seq;
    // kernels: the append waits for the flag itself; the slot's last output
    // must have left d_out (normally long done: then no wait is queued)
    const cudaError_t q = cudaEventQuery(slot->out);
    if (q == cudaErrorNotReady) {
      (void)cudaGetLastError();   // "not ready" is recorded as the last error: clear it
      if (cudaStreamWaitEvent(s_run, slot->out, 0) != cudaSuccess)
        return step_fail(HB_ERR_CUDA, "ordering the kernels failed");
    } else if (q != cudaSuccess) {
      return step_fail(HB_ERR_CUDA, "querying the slot's output copy failed");
    }
    s = hb::internal_kv_append(&b, d_in + off[1], d_in + off[2], k_cache, v_cache, stream,
                               slot->flag, seq);
    if (s != HB_OK) return s;
    // the chunks read their new rows from d_in, not after the append
    s = hb_attention_new_kv(&b, buf->h_plan, d_in + off[0], d_in + off[1], d_in + off[2], k_cache,
                            v_cache, softmax_scale, buf->d_out, buf->d_workspace, stream);
    if (s != HB_OK) return s;
    if (cudaEventRecord(slot->done, s_run) != cudaSuccess)
      return step_fail(HB_ERR_CUDA, "recording the kernels' end failed");
    // output: after the kernels
    const size_t out_bytes =
        (size_t)shape->total_q * (size_t)shape->num_q_heads * (size_t)shape->head_dim * 2;
    if (cudaStreamWaitEvent(s_out, slot->done, 0) != cudaSuccess ||
        cudaMemcpyAsync(buf->h_out, buf->d_out, out_bytes, cudaMemcpyDeviceToHost, s_out) !=
            cudaSuccess ||
        cudaEventRecord(slot->out, s_out) != cudaSuccess)
      return step_fail(HB_ERR_CUDA, "the output copy failed");
    return hb::internal_ok();
  } catch (...) {
    return step_fail(HB_ERR_CUDA, "unexpected exception in hb_step");
  }
}

}  // extern "C"
