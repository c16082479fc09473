// api.cu -- the C ABI of libhb (declared in include/hb.h): argument checks,
// the host-side plan, TMA descriptors, kernel launches, the device error word
// and launch timing.  Every exported function catches everything: no C++
// exception crosses the boundary.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <unordered_map>
#include <string>
#include <vector>

#include "hb.h"
#include "decode_plan.h"
#include "hb_internal.h"

__device__ int g_hb_device_error = 0;

namespace hb {
cudaError_t launch_kv_append(const AppendParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_linear(const LinearParams& p, const CUtensorMap& xmap, const CUtensorMap& wmap,
                          int num_sms, cudaStream_t stream);
int linear_w_box_rows();
int linear_split(int M, int N, int K, int epilogue, int num_sms, int* kb_per_piece);
size_t linear_workspace_bytes(int M, int N, int K, int epilogue, int num_sms);
size_t linear_counter_bytes();
cudaError_t launch_wait_timeout(int* dev_error, cudaStream_t stream);
cudaError_t launch_flag_timeout(int* dev_error, cudaStream_t stream);
cudaError_t launch_attention(const DecodeParams& dec, int decode_grid, const ChunkParams& chk,
                             int head_dim, const CUtensorMap& dec_k, const CUtensorMap& dec_v,
                             const CUtensorMap& chunk_q, const CUtensorMap& chunk_k,
                             const CUtensorMap& chunk_v, const CUtensorMap& chunk_knew,
                             const CUtensorMap& chunk_vnew, const void* k_cache,
                             const void* v_cache, cudaStream_t stream, bool early,
                             int pairs_mode);
}  // namespace hb

using namespace hb;

namespace {

thread_local std::string t_err;

hb_status fail(hb_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return s;
}

hb_status ok() {
  t_err.clear();
  return HB_OK;
}

hb_status cuda_fail(cudaError_t e, const char* what) {
  return fail(HB_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

std::atomic<int64_t> g_launches{0};

// ---------------------------------------------------------------- per device
struct DevState {
  bool ready = false;
  int* err = nullptr;
  int num_sms = 0;
};
std::mutex g_dev_mu;
DevState g_dev[64];

hb_status device_state(DevState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(HB_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevState& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_hb_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    d.err = static_cast<int*>(p);
    d.ready = true;
  }
  *out = &d;
  return HB_OK;
}

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

hb_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(HB_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  return HB_OK;
}

hb_status encode_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides_bytes, const cuuint32_t* box,
                     const char* what) {
  cuuint32_t elem[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                        const_cast<void*>(base), dims, strides_bytes, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HB_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return HB_OK;
}

// ---------------------------------------------------------------- timing
struct TimingRec {
  cudaEvent_t a, b;
  int kernel;
};
std::mutex g_time_mu;
bool g_timing = false;
std::vector<TimingRec> g_recs;
std::vector<cudaEvent_t> g_event_pool;
constexpr size_t kMaxTimingRecs = 1 << 14;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Bracket one launch with events when timing is on.
struct LaunchTimer {
  TimingRec rec{};
  bool on = false;
  cudaStream_t s;
  LaunchTimer(int kernel, cudaStream_t stream) : s(stream) {
    std::lock_guard<std::mutex> lk(g_time_mu);
    if (!g_timing || g_recs.size() >= kMaxTimingRecs) return;
    rec.a = pool_event();
    rec.b = pool_event();
    rec.kernel = kernel;
    if (!rec.a || !rec.b) return;
    on = cudaEventRecord(rec.a, s) == cudaSuccess;
  }
  void done() {
    if (!on) return;
    if (cudaEventRecord(rec.b, s) != cudaSuccess) return;
    std::lock_guard<std::mutex> lk(g_time_mu);
    g_recs.push_back(rec);
  }
};

// ---------------------------------------------------------------- checks
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

hb_status check_batch(const hb_batch* b) {
  if (!b) return fail(HB_ERR_INVALID_ARG, "batch is NULL");
  if (b->num_seqs < 0 || b->total_q < 0)
    return fail(HB_ERR_SHAPE, "num_seqs (%d) and total_q (%d) must be >= 0", b->num_seqs, b->total_q);
  if (b->total_q > 0 && b->num_seqs == 0)
    return fail(HB_ERR_SHAPE, "total_q > 0 with no sequences");
  if (b->page_size != kPageSize)
    return fail(HB_ERR_UNSUPPORTED, "page_size %d (only 16 is built)", b->page_size);
  if (b->head_dim != 64 && b->head_dim != 128)
    return fail(HB_ERR_UNSUPPORTED, "head_dim %d (64 or 128 are built)", b->head_dim);
  if (b->num_q_heads <= 0 || b->num_kv_heads <= 0 || b->num_q_heads % b->num_kv_heads)
    return fail(HB_ERR_SHAPE, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                b->num_q_heads, b->num_kv_heads);
  const int g = b->num_q_heads / b->num_kv_heads;
  if (g > kMaxGroup) return fail(HB_ERR_UNSUPPORTED, "group size %d > %d", g, kMaxGroup);
  if (b->num_kv_heads > kDecodeKvhBlock && b->num_kv_heads % kDecodeKvhBlock)
    return fail(HB_ERR_UNSUPPORTED, "num_kv_heads %d: more than 8 must be a multiple of 8",
                b->num_kv_heads);
  if (b->max_pages_per_seq <= 0 || b->num_pages <= 0)
    return fail(HB_ERR_SHAPE, "max_pages_per_seq and num_pages must be > 0");
  if ((int64_t)b->num_pages * kPageSize > 0x7fffffffLL)
    return fail(HB_ERR_UNSUPPORTED, "num_pages %d too large", b->num_pages);
  if (b->sliding_window < 0) return fail(HB_ERR_SHAPE, "sliding_window %d < 0", b->sliding_window);
  if (b->reserved != 0) return fail(HB_ERR_INVALID_ARG, "hb_batch.reserved must be 0");
  if (b->num_seqs > 0 && (!b->cu_q_len || !b->context_len || !b->block_table))
    return fail(HB_ERR_INVALID_ARG, "cu_q_len, context_len and block_table must be non-NULL");
  return HB_OK;
}

hb_status check_ptr(const void* p, const char* name) {
  if (!p) return fail(HB_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(HB_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return HB_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A named range on the profiler's host timeline around each entry point of
// the hot path (NVTX; a no-op unless a profiling tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};


// ---------------------------------------------------------------- plan scratch
struct DurGroup {
  double d;       // duration of each piece (us)
  int32_t count;  // pieces of that duration
};
struct FreeAt {
  double t;       // an SM frees up at t
  int32_t count;  // SMs that free up then
};

// Working arrays of hb_plan, kept per host thread so that their capacity
// carries over from call to call.
struct PlanScratch {
  std::vector<ChunkItem> raw, chk;
  std::vector<int32_t> count;
  std::vector<int32_t> dur_count;
  std::vector<int32_t> hist;
  std::vector<DurGroup> groups;
  std::vector<FreeAt> free_at, next, fresh;
  std::vector<DecodeItem> dec;
  std::vector<int32_t> cta_off;
  std::vector<double> t_end;
};

PlanScratch& plan_scratch() {
  thread_local PlanScratch ps;
  return ps;
}

// Stable sort of `in` into `out` by key(x) in 0..kmax, largest key first.
template <class T, class Key>
void counting_sort_desc(const std::vector<T>& in, std::vector<T>& out, std::vector<int32_t>& cnt,
                        int kmax, Key key) {
  cnt.assign((size_t)kmax + 2, 0);
  for (const T& x : in) ++cnt[key(x)];
  int32_t run = 0;
  for (int k = kmax; k >= 0; --k) {
    const int32_t c = cnt[k];
    cnt[k] = run;
    run += c;
  }
  out.resize(in.size());
  for (const T& x : in) out[cnt[key(x)]++] = x;
}

// End time of a launch whose pieces (ps.groups: durations, longest first,
// with their counts) start one after another, each on the SM that frees up
// first; G of the num_sms SMs are busy until td, the others free at 0.  The
// same end as placing the pieces one by one with a heap of SM free times,
// computed on (time, count) runs: within a run of equal durations the next
// piece takes the earlier of the oldest free time left and the oldest time
// freed by the run itself, both of which come in ascending order.
double simulate_dispatch(PlanScratch& ps, int num_sms, int G, double td) {
  std::vector<FreeAt>& F = ps.free_at;
  F.clear();
  if (G < num_sms) F.push_back({0.0, num_sms - G});
  if (G > 0) F.push_back({td, G});
  double end = td;
  for (const DurGroup& grp : ps.groups) {
    std::vector<FreeAt>& Q = ps.fresh;   // times freed by this run, ascending
    Q.clear();
    size_t i1 = 0, i2 = 0;
    int32_t left = grp.count;
    double last = 0.0;
    while (left > 0) {
      const bool from_f = i1 < F.size() && (i2 >= Q.size() || F[i1].t <= Q[i2].t);
      FreeAt* src = from_f ? &F[i1] : &Q[i2];
      const int32_t k = std::min(src->count, left);
      const double t = src->t;
      src->count -= k;               // (before the push below can move Q)
      if (src->count == 0) {
        if (from_f) ++i1; else ++i2;
      }
      last = t;
      left -= k;
      Q.push_back({t + grp.d, k});
    }
    end = std::max(end, last + grp.d);
    // the free times left: the rest of F merged with the rest of Q
    std::vector<FreeAt>& M = ps.next;
    M.clear();
    while (i1 < F.size() || i2 < Q.size()) {
      const bool from_f = i1 < F.size() && (i2 >= Q.size() || F[i1].t <= Q[i2].t);
      const FreeAt x = from_f ? F[i1++] : Q[i2++];
      if (x.count == 0) continue;
      if (!M.empty() && M.back().t == x.t) M.back().count += x.count;
      else M.push_back(x);
    }
    F.swap(M);
  }
  return end;
}
}  // namespace

// ---------------------------------------------------------------- internal
// Hooks for other translation units of the library (not part of the ABI).
namespace hb {

hb_status internal_fail(hb_status s, const char* msg) { return fail(s, "%s", msg); }

hb_status internal_ok() { return ok(); }

hb_status internal_check_batch(const hb_batch* b) { return check_batch(b); }

hb_status internal_device(int** err, int* num_sms) {
  DevState* d = nullptr;
  hb_status s = device_state(&d);
  if (s != HB_OK) return s;
  *err = d->err;
  *num_sms = d->num_sms;
  return HB_OK;
}

// TMA maps of the decode kernel over the K and V pools.
hb_status internal_decode_maps(const hb_batch* b, int kvhb, const void* k_cache,
                               const void* v_cache, CUtensorMap* kmap, CUtensorMap* vmap) {
  hb_status s = get_encoder();
  if (s != HB_OK) return s;
  const int Hkv = b->num_kv_heads, D = b->head_dim;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPageSize, (cuuint64_t)Hkv,
                              (cuuint64_t)b->num_pages};
  const cuuint64_t strides[3] = {(cuuint64_t)Hkv * D * 2, (cuuint64_t)D * 2,
                                 (cuuint64_t)kPageSize * Hkv * D * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)kPageSize, (cuuint32_t)kvhb, 1};
  if ((s = encode_map(kmap, k_cache, 4, dims, strides, box, "decode K")) != HB_OK) return s;
  return encode_map(vmap, v_cache, 4, dims, strides, box, "decode V");
}

void internal_count_launch() { g_launches.fetch_add(1); }

// ---------------------------------------------------------------- launch order
// The library's last launch on each stream.  The attention kernel may read
// the cache pages that hold none of its batch's new tokens before the grid
// before it has finished (it waits only before the pages with new tokens)
// when that grid is hb_kv_append of the same batch: that append writes only
// those tokens.  After any other launch of this library it waits first.
// Work of other libraries between the two is launched without programmatic
// serialization, so it starts only after the append has finished and does
// not release the attention early: a stale record is safe.
namespace {
enum LaunchKind { kOtherLaunch = 0, kAppendLaunch = 1 };
struct LastLaunch {
  int kind = kOtherLaunch;
  const void *cu = nullptr, *ctx = nullptr, *bt = nullptr, *kc = nullptr, *vc = nullptr;
};
std::mutex g_last_mu;
std::unordered_map<void*, LastLaunch> g_last;
void note_launch(void* stream, const LastLaunch& l) {
  std::lock_guard<std::mutex> lk(g_last_mu);
  g_last[stream] = l;
}
bool follows_own_append(void* stream, const hb_batch* b, const void* kc, const void* vc) {
  std::lock_guard<std::mutex> lk(g_last_mu);
  auto it = g_last.find(stream);
  if (it == g_last.end()) return false;
  const LastLaunch& l = it->second;
  return l.kind == kAppendLaunch && l.cu == b->cu_q_len && l.ctx == b->context_len &&
         l.bt == b->block_table && l.kc == kc && l.vc == vc;
}
}  // namespace

void internal_note_other_launch(void* stream) { note_launch(stream, LastLaunch{}); }

// hb_kv_append, optionally gated on a flag raised by a copy on another
// stream (defined below)
hb_status internal_kv_append(const hb_batch* batch, const void* k_new, const void* v_new,
                             void* k_cache, void* v_cache, void* stream,
                             const uint32_t* ready_flag, uint32_t ready_value);

// hb_attention, optionally reading the new tokens' K/V from k_new / v_new
// (defined below)
hb_status internal_attention(const hb_batch* batch, const void* h_plan, const void* q,
                             const void* k_new, const void* v_new, const void* k_cache,
                             const void* v_cache, float softmax_scale, void* out,
                             void* d_workspace, void* stream);

}  // namespace hb

// =========================================================================
extern "C" {

const char* hb_last_error(void) { return t_err.c_str(); }

const char* hb_status_string(hb_status s) {
  switch (s) {
    case HB_OK: return "HB_OK";
    case HB_ERR_INVALID_ARG: return "HB_ERR_INVALID_ARG";
    case HB_ERR_SHAPE: return "HB_ERR_SHAPE";
    case HB_ERR_UNSUPPORTED: return "HB_ERR_UNSUPPORTED";
    case HB_ERR_WORKSPACE: return "HB_ERR_WORKSPACE";
    case HB_ERR_CUDA: return "HB_ERR_CUDA";
    case HB_ERR_DEVICE_INDEX: return "HB_ERR_DEVICE_INDEX";
    case HB_ERR_TIMEOUT: return "HB_ERR_TIMEOUT";
    case HB_ERR_OUT_OF_PAGES: return "HB_ERR_OUT_OF_PAGES";
  }
  return "HB_ERR_UNKNOWN";
}

hb_status hb_kv_append(const hb_batch* batch, const void* k_new, const void* v_new,
                       void* k_cache, void* v_cache, void* stream) {
  return hb::internal_kv_append(batch, k_new, v_new, k_cache, v_cache, stream, nullptr, 0);
}

}  // extern "C"

hb_status hb::internal_kv_append(const hb_batch* batch, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, void* stream,
                                 const uint32_t* ready_flag, uint32_t ready_value) {
  NvtxRange range("hb_kv_append");
  try {
    hb_status s = check_batch(batch);
    if (s != HB_OK) return s;
    if (batch->total_q == 0) return ok();
    if ((s = check_ptr(k_new, "k_new")) != HB_OK) return s;
    if ((s = check_ptr(v_new, "v_new")) != HB_OK) return s;
    if ((s = check_ptr(k_cache, "k_cache")) != HB_OK) return s;
    if ((s = check_ptr(v_cache, "v_cache")) != HB_OK) return s;
    DevState* dev = nullptr;
    if ((s = device_state(&dev)) != HB_OK) return s;
    AppendParams p{};
    p.cu_q_len = batch->cu_q_len;
    p.context_len = batch->context_len;
    p.block_table = batch->block_table;
    p.num_seqs = batch->num_seqs;
    p.total_q = batch->total_q;
    p.max_pages_per_seq = batch->max_pages_per_seq;
    p.num_pages = batch->num_pages;
    p.row_vec16 = batch->num_kv_heads * batch->head_dim * 2 / 16;
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.k_cache = static_cast<uint16_t*>(k_cache);
    p.v_cache = static_cast<uint16_t*>(v_cache);
    p.dev_error = dev->err;
    p.ready_flag = ready_flag;
    p.ready_value = ready_value;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    LaunchTimer t(0, st);
    cudaError_t e = launch_kv_append(p, dev->num_sms, st);
    t.done();
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    LastLaunch rec;
    rec.kind = kAppendLaunch;
    rec.cu = batch->cu_q_len;
    rec.ctx = batch->context_len;
    rec.bt = batch->block_table;
    rec.kc = k_cache;
    rec.vc = v_cache;
    note_launch(stream, rec);
    g_launches.fetch_add(1);
    return ok();
  } catch (...) {
    return fail(HB_ERR_CUDA, "unexpected exception in hb_kv_append");
  }
}

extern "C" {

size_t hb_linear_workspace_size(int32_t M, int32_t N, int32_t K, int32_t epilogue,
                                int32_t num_sms) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 64 || N % 256 || num_sms <= 0 ||
      epilogue < HB_LINEAR_STORE || epilogue > HB_LINEAR_RESIDUAL)
    return 0;
  return linear_workspace_bytes(M, N, K, epilogue, num_sms);
}

hb_status hb_linear(const void* x, const void* w, int32_t M, int32_t N, int32_t K,
                    int32_t epilogue, const hb_linear_out* out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  NvtxRange range("hb_linear");
  try {
    if (!out) return fail(HB_ERR_INVALID_ARG, "out is NULL");
    if (epilogue < HB_LINEAR_STORE || epilogue > HB_LINEAR_RESIDUAL)
      return fail(HB_ERR_INVALID_ARG, "unknown epilogue %d", epilogue);
    if (M < 0 || N <= 0 || K <= 0) return fail(HB_ERR_SHAPE, "M %d, N %d, K %d", M, N, K);
    if (K % 64) return fail(HB_ERR_SHAPE, "K (%d) must be a multiple of 64", K);
    hb_status s;
    if ((s = check_ptr(x, "x")) != HB_OK) return s;
    if ((s = check_ptr(w, "w")) != HB_OK) return s;
    LinearParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.epilogue = epilogue;
    if (epilogue == HB_LINEAR_GATED) {
      if (N % 256) return fail(HB_ERR_SHAPE, "gated: N = 2F (%d) must be a multiple of 256", N);
      p.F = N / 2;
      if (out->cols[0] != p.F || out->cols[1] != 0 || out->cols[2] != 0)
        return fail(HB_ERR_SHAPE, "gated: cols must be {F, 0, 0} with F = %d", p.F);
    } else {
      if (N % 256) return fail(HB_ERR_SHAPE, "N (%d) must be a multiple of 256", N);
      int64_t sum = 0;
      for (int i = 0; i < 3; ++i) {
        if (out->cols[i] < 0 || out->cols[i] % 256)
          return fail(HB_ERR_SHAPE, "cols[%d] = %d: multiples of 256 needed", i, out->cols[i]);
        sum += out->cols[i];
      }
      if (sum != N) return fail(HB_ERR_SHAPE, "cols sum to %lld, N is %d", (long long)sum, N);
    }
    for (int i = 0; i < 3; ++i) {
      if (out->cols[i] == 0) continue;
      if ((s = check_ptr(out->y[i], "out->y[i]")) != HB_OK) return s;
      p.y[i] = static_cast<uint16_t*>(out->y[i]);
      p.seg_cols[i] = out->cols[i];
    }
    if (M == 0) return ok();
    DevState* dev = nullptr;
    if ((s = device_state(&dev)) != HB_OK) return s;
    if ((s = get_encoder()) != HB_OK) return s;
    p.dev_error = dev->err;
    // split-K when the tiles are few and the caller gave room for it
    p.split = 1;
    p.kb_per_piece = K / 64;
    const size_t need = linear_workspace_bytes(M, N, K, epilogue, dev->num_sms);
    if (need > 0 && workspace != nullptr && workspace_bytes >= need &&
        (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0) {
      int kbp = 0;
      p.split = linear_split(M, N, K, epilogue, dev->num_sms, &kbp);
      p.kb_per_piece = kbp;
      p.tile_counters = static_cast<int32_t*>(workspace);
      p.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + linear_counter_bytes());
    }
    CUtensorMap xmap, wmap;
    const cuuint64_t xdims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t xstr[1] = {(cuuint64_t)K * 2};
    const cuuint32_t xbox[2] = {64, 128};
    if ((s = encode_map(&xmap, x, 2, xdims, xstr, xbox, "linear x")) != HB_OK) return s;
    const cuuint64_t wdims[2] = {(cuuint64_t)K, (cuuint64_t)N};
    const cuuint32_t wbox[2] = {64, (cuuint32_t)linear_w_box_rows()};
    if ((s = encode_map(&wmap, w, 2, wdims, xstr, wbox, "linear w")) != HB_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    LaunchTimer t(2, st);
    cudaError_t e = launch_linear(p, xmap, wmap, dev->num_sms, st);
    t.done();
    if (e != cudaSuccess) return cuda_fail(e, "linear launch");
    note_launch(stream, LastLaunch{});
    g_launches.fetch_add(1);
    return ok();
  } catch (...) {
    return fail(HB_ERR_CUDA, "unexpected exception in hb_linear");
  }
}

hb_status hb_plan(const hb_batch* batch, const int32_t* h_q_len,
                  const int32_t* h_context_len, int32_t num_sms, void* h_plan,
                  size_t* plan_bytes, void* d_workspace, size_t* workspace_bytes,
                  void* stream) {
  NvtxRange range("hb_plan");
  try {
    hb_status s = check_batch(batch);
    if (s != HB_OK) return s;
    if (!plan_bytes || !workspace_bytes)
      return fail(HB_ERR_INVALID_ARG, "plan_bytes and workspace_bytes must be non-NULL");
    if (num_sms <= 0) return fail(HB_ERR_INVALID_ARG, "num_sms must be > 0");
    const int S = batch->num_seqs;
    if (S > 0 && (!h_q_len || !h_context_len))
      return fail(HB_ERR_INVALID_ARG, "h_q_len and h_context_len must be non-NULL");
    const int Hq = batch->num_q_heads, Hkv = batch->num_kv_heads, D = batch->head_dim;
    const int g = Hq / Hkv;
    const int W = batch->sliding_window;
    const int64_t max_ctx = (int64_t)batch->max_pages_per_seq * kPageSize;
    int64_t tq = 0;
    for (int i = 0; i < S; ++i) {
      if (h_q_len[i] < 1 || h_q_len[i] > h_context_len[i])
        return fail(HB_ERR_SHAPE, "row %d: q_len %d, context_len %d (need 1 <= q_len <= context_len)",
                    i, h_q_len[i], h_context_len[i]);
      if (h_context_len[i] > max_ctx)
        return fail(HB_ERR_SHAPE, "row %d: context_len %d exceeds max_pages_per_seq * 16", i,
                    h_context_len[i]);
      tq += h_q_len[i];
    }
    if (tq != batch->total_q)
      return fail(HB_ERR_SHAPE, "sum of q_len (%lld) != total_q (%d)", (long long)tq, batch->total_q);

    const int kvhb = std::min(Hkv, kDecodeKvhBlock);
    const int n_blocks = Hkv / kvhb;
    // all working arrays live in per-thread storage that keeps its capacity
    // from call to call: a plan of a batch shaped like the last one
    // allocates nothing
    PlanScratch& ps = plan_scratch();

    // ---- chunk items: rows with q_len > 1, (kv head, query tile or pair of
    // query tiles)
    const int tpt = kChunkRows / g;
    int64_t n_tiles_total = 0;
    for (int i = 0; i < S; ++i)
      if (h_q_len[i] > 1) n_tiles_total += (int64_t)((h_q_len[i] + tpt - 1) / tpt) * Hkv;
    auto key_tiles = [](const ChunkItem& c) { return c.kv_tiles - c.kv_begin; };
    // the items of one layout (tpi query tiles per item) into ps.chk,
    // longest first (stable: ties keep the order row, kv head, t0).  An
    // item's key-tile count depends on its row and t0 only, so the counts
    // are taken once per (row, t0), Hkv items each, and every item is then
    // written once, straight into its place.
    auto build_items = [&](int tpi) {
      const int item_tokens = tpi * tpt;
      // key-tile range [*kb, return) of the item of row i starting at t0
      auto range_of = [&](int i, int t0, int* kb) {
        const int off = h_context_len[i] - h_q_len[i];
        const int ntok = std::min(item_tokens, h_q_len[i] - t0);
        // with a sliding window the first row sees keys from off+t0-W+1 on
        *kb = W > 0 ? std::max(0, off + t0 - W + 1) / kChunkKeys : 0;
        return (off + t0 + ntok + kChunkKeys - 1) / kChunkKeys;
      };
      int key_max = 0;
      size_t n = 0;
      for (int i = 0; i < S; ++i) {
        if (h_q_len[i] == 1) continue;
        for (int t0 = 0; t0 < h_q_len[i]; t0 += item_tokens) {
          int kb;
          key_max = std::max(key_max, range_of(i, t0, &kb) - kb);
          n += (size_t)Hkv;
        }
      }
      ps.count.assign((size_t)key_max + 2, 0);
      for (int i = 0; i < S; ++i) {
        if (h_q_len[i] == 1) continue;
        for (int t0 = 0; t0 < h_q_len[i]; t0 += item_tokens) {
          int kb;
          ps.count[range_of(i, t0, &kb) - kb] += Hkv;
        }
      }
      int32_t run = 0;
      for (int k = key_max; k >= 0; --k) {
        const int32_t c = ps.count[k];
        ps.count[k] = run;
        run += c;
      }
      ps.chk.resize(n);
      int32_t q0 = 0;
      for (int i = 0; i < S; q0 += h_q_len[i], ++i) {
        if (h_q_len[i] == 1) continue;
        // the last item of a row may be short (a pair's second tile short
        // or empty)
        for (int kvh = 0; kvh < Hkv; ++kvh)
          for (int t0 = 0; t0 < h_q_len[i]; t0 += item_tokens) {
            int kb;
            const int kt = range_of(i, t0, &kb);
            ps.chk[ps.count[kt - kb]++] =
                ChunkItem{i, kvh, t0, std::min(item_tokens, h_q_len[i] - t0), kt, q0, h_q_len[i],
                          h_context_len[i], kb, 0, 1, 0, 0, 0, 0, 0};
          }
      }
    };

    // ---- cost model, in microseconds, from rates measured on GB300.  The
    // attention kernel runs decode CTAs and chunk CTAs side by side (one CTA
    // per SM); SMs that end their decode range go on to chunk items.  With G
    // decode CTAs, decode takes its bytes over min(HBM rate, G x one SM's
    // stream rate); everything ends no earlier than (chunk work + G x decode
    // time) / SMs, nor before the longest chunk item.  That estimate is flat
    // over a range of G whose ends it knows only roughly, so the middle of
    // the range within 2% of the best is taken.  A pair of query tiles
    // shares its page gather, so it costs 1.6x one tile, not 2x.  A split
    // piece pays its own setup (barriers, Q load, pipeline fill) and its
    // publish-and-merge: per-CTA timelines show split pair pieces at 1.9-2.2
    // us per key tile against 1.56 for whole pairs, and on the chunk-only
    // sweep (8192-token prompt, chunks of 256 / 512 / 1024) a piece cost of
    // 10 us gave 1.310 / 0.804 / 0.584 ms against 1.376 / 0.833 / 0.637 ms
    // at 3 us (6: 1.311 / 0.814 / 0.586, 15: 1.298 / 0.824 / 0.585), the
    // batches with decode rows unchanged.
    constexpr double kHbmBytesPerUs = 7.0e6;      // whole-GPU HBM stream
    constexpr double kSmBytesPerUs = 8.5e4;       // one SM's stream ceiling
    constexpr double kPairTileUs = 2.0;           // 2-tile item x one key tile
    constexpr double kSingleTileUs = 1.25;        // 1-tile item x one key tile
    constexpr double kPieceUs = 10.0;             // extra cost of one split piece
    constexpr int kMinPieceTiles = 4;             // key tiles per split piece (min)
    double decode_bytes = 0.0;
    for (int i = 0; i < S; ++i)
      if (h_q_len[i] == 1)
        decode_bytes += (double)(W > 0 ? std::min(h_context_len[i], W) : h_context_len[i]) * Hkv * D * 4.0;
    auto t_decode = [&](int G) {
      return decode_bytes / std::min(kHbmBytesPerUs, G * kSmBytesPerUs);
    };
    // t(G) falls while G SMs cannot stream at the HBM rate (G x one SM's
    // rate below it: t_decode shrinks, G x t_decode stays) and rises after
    // (t_decode fixed, G x t_decode grows), so each side is searched by
    // bisection instead of evaluating every G
    auto pick_decode = [&](double chunk_us, double max_item_us) -> int {
      if (decode_bytes <= 0.0) return 0;
      if (chunk_us <= 0.0) return num_sms;
      auto t_of = [&](int G) {
        const double td = t_decode(G);
        return std::max({td, (chunk_us + G * td) / num_sms, max_item_us});
      };
      // the last G whose SMs together stream below the HBM rate
      int gs = std::min(num_sms, std::max(1, (int)(kHbmBytesPerUs / kSmBytesPerUs)));
      while (gs > 1 && gs * kSmBytesPerUs >= kHbmBytesPerUs) --gs;
      while (gs < num_sms && (gs + 1) * kSmBytesPerUs < kHbmBytesPerUs) ++gs;
      const double best = std::min(t_of(gs), gs < num_sms ? t_of(gs + 1) : 1e300);
      const double lim = 1.02 * best;
      // lo: the first G in 1..gs with t(G) <= lim (t non-increasing there)
      int a = 1, b = gs;
      if (t_of(gs) > lim) a = gs + 1;   // none on this side
      while (a < b) {
        const int m = (a + b) / 2;
        if (t_of(m) <= lim) b = m; else a = m + 1;
      }
      const int lo = a;
      // hi: the last G in gs+1..num_sms with t(G) <= lim (t non-decreasing)
      int hi = lo <= gs ? gs : lo;
      if (gs < num_sms && t_of(gs + 1) <= lim) {
        int c = gs + 1, d = num_sms;
        while (c < d) {
          const int m = (c + d + 1) / 2;
          if (t_of(m) <= lim) c = m; else d = m - 1;
        }
        hi = c;
      }
      return (lo + hi) / 2;
    };
    // pieces per item when each piece holds about L key tiles
    auto pieces_of = [&](int kv, int L) {
      int n = std::min(kMaxChunkSplits, (kv + L - 1) / L);
      return std::max(1, std::min(n, kv / kMinPieceTiles));
    };

    // ---- split-KV: when the items are too few to fill the SMs, an item's
    // key range may be cut into up to kMaxChunkSplits pieces (each its own
    // CTA, merged by the last to finish).  The piece length is the one with
    // the earliest estimated end among a few candidates (no split included);
    // the end is that of CTAs started in index order on the SM that frees up
    // first, the G decode CTAs first, holding their SMs for the decode time
    // (simulate_dispatch).  Returns that end; *out_L = 0 for no split.
    auto search_split = [&](double tile_us, int* out_L) -> double {
      *out_L = 0;
      if (ps.chk.empty()) return 0.0;
      // more items than two waves: no split is allowed (every candidate
      // below gives up at once), and the pair layout is taken without a
      // comparison, so the end time is not needed
      if ((int64_t)ps.chk.size() > 2LL * num_sms) return 0.0;
      const int kmax = key_tiles(ps.chk.front());
      // items by key-tile count: a candidate costs what the distinct counts
      // cost, not what the items do
      ps.hist.assign((size_t)kmax + 1, 0);
      for (const ChunkItem& c : ps.chk) ++ps.hist[key_tiles(c)];
      double best_t = 1e300;
      int prev_L = -1;
      for (int n = 1; n <= kMaxChunkSplits; ++n) {
        const int L = (kmax + n - 1) / n;
        if (L == prev_L || (n > 1 && L < kMinPieceTiles)) continue;
        prev_L = L;
        // pieces counted per (length, split) class
        ps.dur_count.assign(2 * (size_t)(kmax + 1), 0);
        int64_t n_pieces = 0;
        double sum = 0.0, mx = 0.0;
        bool too_many = false;
        for (int kv = kmax; kv >= 0 && !too_many; --kv) {
          const int32_t items = ps.hist[kv];
          if (!items) continue;
          const int np = n == 1 ? 1 : pieces_of(kv, L);
          for (int k = 0; k < np; ++k) {
            const int len = (k + 1) * kv / np - k * kv / np;
            const double d = len * tile_us + (np > 1 ? kPieceUs : 0.0);
            ps.dur_count[2 * (size_t)len + (np > 1 ? 1 : 0)] += items;
            sum += items * d;
            mx = std::max(mx, d);
          }
          n_pieces += (int64_t)np * items;
          too_many = n > 1 && n_pieces > 2LL * num_sms;
        }
        if (too_many) break;   // at most two waves
        ps.groups.clear();
        for (int len = 0; len <= kmax; ++len)
          for (int sp = 0; sp < 2; ++sp) {
            const int32_t cnt = ps.dur_count[2 * (size_t)len + sp];
            if (cnt) ps.groups.push_back({len * tile_us + (sp ? kPieceUs : 0.0), cnt});
          }
        std::sort(ps.groups.begin(), ps.groups.end(),
                  [](const DurGroup& a, const DurGroup& b) { return a.d > b.d; });
        const int G = pick_decode(sum, mx);
        const double t = simulate_dispatch(ps, num_sms, G, G > 0 ? t_decode(G) : 0.0);
        if (t < 0.97 * best_t) {   // a split has to pay for itself clearly
          best_t = t;
          *out_L = n == 1 ? 0 : L;
        }
      }
      return best_t;
    };
    // Layout: pairs of query tiles, which share every K/V tile they gather,
    // or -- when the tiles are too few to fill the GPU twice -- whichever of
    // pairs and single tiles (each with its best split) ends earlier.
    int tiles_per_item = 2, best_L = 0;
    ps.chk.clear();
    if (n_tiles_total > 0) {
      double t_single = 1e300;
      int L_single = 0;
      if (n_tiles_total < 2LL * num_sms) {
        build_items(1);
        t_single = search_split(kSingleTileUs, &L_single);
      }
      build_items(2);
      int L_pair = 0;
      const double t_pair = search_split(kPairTileUs, &L_pair);
      if (t_single < t_pair) {
        tiles_per_item = 1;
        best_L = L_single;
        build_items(1);
      } else {
        best_L = L_pair;
      }
    }
    const double tile_us = tiles_per_item == 2 ? kPairTileUs : kSingleTileUs;
    int n_cslots = 0, n_cmerge = 0;
    if (best_L > 0) {
      ps.raw.clear();
      int piece_max = 0;
      for (ChunkItem c : ps.chk) {
        const int kv = key_tiles(c);
        const int kb0 = c.kv_begin;
        const int np = pieces_of(kv, best_L);
        // a split pair keeps one partial state per tile and piece
        const int tiles = c.ntok > tpt ? 2 : 1;
        c.n_splits = np;
        c.slot = np > 1 ? n_cslots : 0;
        c.merge_id = np > 1 ? n_cmerge : 0;
        for (int k = 0; k < np; ++k) {
          c.split = k;
          c.kv_begin = kb0 + k * kv / np;
          c.kv_tiles = kb0 + (k + 1) * kv / np;
          piece_max = std::max(piece_max, key_tiles(c));
          ps.raw.push_back(c);
        }
        if (np > 1) {
          n_cslots += np * tiles;
          n_cmerge += 1;
        }
      }
      // longest first, so that short pieces fill the end of the launch
      counting_sort_desc(ps.raw, ps.chk, ps.count, piece_max, key_tiles);
    }
    // (without a split every item is one piece and the order stands)
    double chunk_us = 0.0, max_item_us = 0.0;
    for (const ChunkItem& c : ps.chk) {
      const double us = (c.kv_tiles - c.kv_begin) * tile_us + (c.n_splits > 1 ? kPieceUs : 0.0);
      chunk_us += us;
      max_item_us = std::max(max_item_us, us);
    }
    const int decode_ctas = pick_decode(chunk_us, max_item_us);

    // ---- decode items: the decode rows' pages, end to end, cut into one
    // equal contiguous range per CTA, each range cut at row boundaries
    int64_t n_dec_rows = 0;
    for (int i = 0; i < S; ++i)
      if (h_q_len[i] == 1) ++n_dec_rows;
    // intervals: one static range per decode CTA.  A dynamic tail (short
    // intervals claimed from a counter) is supported by partition_decode and
    // the kernel but measured slower on GB300 (Mistral 125 vs 110 us: the
    // extra pieces and merges cost more than the ragged tail), so it is off.
    const int max_intervals = std::max(1, decode_ctas) * (1 + kDynamicPerCta) + 1;
    const int max_dec_items =
        (int)std::min<int64_t>(n_dec_rows * n_blocks + max_intervals + 1, 1 << 30);
    ps.dec.resize(std::max(1, max_dec_items));
    ps.cta_off.resize(max_intervals + 1);
    ps.cta_off[0] = 0;
    DecodePartition part;
    if (!partition_decode(S, h_q_len, h_context_len, n_blocks, kvhb, std::max(1, decode_ctas), 4,
                          ps.dec.data(), (int)ps.dec.size(), ps.cta_off.data(), max_intervals,
                          &part, W, /*dynamic_tail=*/false))
      return fail(HB_ERR_WORKSPACE, "decode partition overflow");
    const size_t n_dec = (size_t)part.n_items;
    const size_t n_chk = ps.chk.size();
    const size_t n_off = (size_t)(part.grid + part.n_dynamic + 1);
    const int n_slots = part.n_slots, n_merge = part.n_merge;

    // ---- sizes
    const size_t offsets_at = n_dec * sizeof(DecodeItem) + n_chk * sizeof(ChunkItem);
    const size_t items_bytes = align_up(offsets_at + n_off * sizeof(int32_t), 256);
    const size_t need_plan = sizeof(PlanHeader) + items_bytes;
    const size_t ws_counters = items_bytes;
    const size_t ws_partial_o = align_up(ws_counters + (size_t)(kCounterMerge0 + n_merge) * 4, 256);
    const size_t ws_partial_ml = align_up(ws_partial_o + (size_t)n_slots * Hq * D * 4, 256);
    const size_t ws_chunk_counters = align_up(ws_partial_ml + (size_t)n_slots * Hq * 8, 256);
    const size_t ws_chunk_o = align_up(ws_chunk_counters + (size_t)n_cmerge * 4, 256);
    const size_t ws_chunk_ml = align_up(ws_chunk_o + (size_t)n_cslots * D * kChunkRows * 4, 256);
    const size_t ws_total =
        std::max<size_t>(256, align_up(ws_chunk_ml + (size_t)n_cslots * 2 * kChunkRows * 4, 256));

    const size_t have_plan = *plan_bytes, have_ws = *workspace_bytes;
    *plan_bytes = need_plan;
    *workspace_bytes = ws_total;
    if (h_plan == nullptr) return ok();  // size query
    if (have_plan < need_plan)
      return fail(HB_ERR_WORKSPACE, "plan buffer has %zu bytes, needs %zu", have_plan, need_plan);
    if (d_workspace != nullptr) {
      if (have_ws < ws_total)
        return fail(HB_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have_ws, ws_total);
      if ((reinterpret_cast<uintptr_t>(d_workspace) & 255u) != 0)
        return fail(HB_ERR_INVALID_ARG, "d_workspace must be 256-byte aligned");
    }

    PlanHeader h{};
    h.magic = kPlanMagic;
    h.version = kPlanVersion;
    h.num_seqs = S;
    h.total_q = batch->total_q;
    h.num_q_heads = Hq;
    h.num_kv_heads = Hkv;
    h.head_dim = D;
    h.page_size = batch->page_size;
    h.max_pages_per_seq = batch->max_pages_per_seq;
    h.num_sms = num_sms;
    h.num_decode_items = (int32_t)n_dec;
    h.num_chunk_items = (int32_t)n_chk;
    h.num_partial_slots = n_slots;
    h.num_merge_counters = n_merge;
    h.decode_grid = part.grid;
    h.num_decode_dynamic = part.n_dynamic;
    {
      // bit 0: every item an unsplit pair; bit 1: some item's first row sees
      // few keys (its P is written in two terms)
      bool pairs = n_chk > 0, few = false;
      for (size_t i = 0; i < n_chk; ++i) {
        const ChunkItem& c = ps.chk[i];
        const int first_keys = c.ctx - c.q_len + c.tok0 + 1;
        pairs = pairs && c.ntok > tpt && c.n_splits == 1;
        few = few || (W > 0 ? std::min(W, first_keys) : first_keys) <= kChunkFewKeys;
      }
      h.chunk_pairs_only = (pairs ? 1 : 0) | (few ? 2 : 0);
    }
    h.ws_decode_offsets = offsets_at;
    h.decode_kvh_block = kvhb;
    h.chunk_tokens_per_tile = tpt;
    h.num_chunk_slots = n_cslots;
    h.num_chunk_merges = n_cmerge;
    h.sliding_window = W;
    h.ws_chunk_counters = ws_chunk_counters;
    h.ws_chunk_o = ws_chunk_o;
    h.ws_chunk_ml = ws_chunk_ml;
    h.items_bytes = items_bytes;
    h.ws_counters = ws_counters;
    h.ws_partial_o = ws_partial_o;
    h.ws_partial_ml = ws_partial_ml;
    h.ws_total = ws_total;
    h.plan_bytes = need_plan;
    uint8_t* hp = static_cast<uint8_t*>(h_plan);
    std::memcpy(hp, &h, sizeof(h));
    uint8_t* items = hp + sizeof(PlanHeader);
    if (n_dec) std::memcpy(items, ps.dec.data(), n_dec * sizeof(DecodeItem));
    if (n_chk) std::memcpy(items + n_dec * sizeof(DecodeItem), ps.chk.data(), n_chk * sizeof(ChunkItem));
    std::memcpy(items + offsets_at, ps.cta_off.data(), n_off * sizeof(int32_t));
    const size_t used = offsets_at + n_off * sizeof(int32_t);
    std::memset(items + used, 0, items_bytes - used);   // alignment padding

    if (d_workspace == nullptr) return ok();  // host plan only
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(d_workspace, items, items_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    e = cudaMemsetAsync(static_cast<uint8_t*>(d_workspace) + ws_counters, 0,
                        ws_partial_o - ws_counters, st);
    if (e != cudaSuccess) return cuda_fail(e, "workspace counter reset");
    if (n_cmerge > 0) {
      e = cudaMemsetAsync(static_cast<uint8_t*>(d_workspace) + ws_chunk_counters, 0,
                          ws_chunk_o - ws_chunk_counters, st);
      if (e != cudaSuccess) return cuda_fail(e, "workspace counter reset");
    }
    return ok();
  } catch (...) {
    return fail(HB_ERR_CUDA, "unexpected exception in hb_plan");
  }
}

hb_status hb_attention(const hb_batch* batch, const void* h_plan, const void* q,
                       const void* k_cache, const void* v_cache, float softmax_scale,
                       void* out, void* d_workspace, void* stream) {
  return hb::internal_attention(batch, h_plan, q, nullptr, nullptr, k_cache, v_cache,
                                softmax_scale, out, d_workspace, stream);
}

hb_status hb_attention_new_kv(const hb_batch* batch, const void* h_plan, const void* q,
                              const void* k_new, const void* v_new, const void* k_cache,
                              const void* v_cache, float softmax_scale, void* out,
                              void* d_workspace, void* stream) {
  if (!k_new || !v_new) return fail(HB_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
  return hb::internal_attention(batch, h_plan, q, k_new, v_new, k_cache, v_cache,
                                softmax_scale, out, d_workspace, stream);
}

}  // extern "C"

// hb_attention; with k_new / v_new (the append's inputs) the chunk CTAs read
// the pages that hold only new tokens from there
hb_status hb::internal_attention(const hb_batch* batch, const void* h_plan, const void* q,
                                 const void* k_new, const void* v_new, const void* k_cache,
                                 const void* v_cache, float softmax_scale, void* out,
                                 void* d_workspace, void* stream) {
  NvtxRange range("hb_attention");
  try {
    hb_status s = check_batch(batch);
    if (s != HB_OK) return s;
    if (!h_plan) return fail(HB_ERR_INVALID_ARG, "h_plan is NULL");
    PlanHeader h;
    std::memcpy(&h, h_plan, sizeof(h));
    if (h.magic != kPlanMagic || h.version != kPlanVersion)
      return fail(HB_ERR_WORKSPACE, "h_plan is not a plan written by hb_plan");
    if (h.num_seqs != batch->num_seqs || h.total_q != batch->total_q ||
        h.num_q_heads != batch->num_q_heads || h.num_kv_heads != batch->num_kv_heads ||
        h.head_dim != batch->head_dim || h.page_size != batch->page_size ||
        h.max_pages_per_seq != batch->max_pages_per_seq ||
        h.sliding_window != batch->sliding_window)
      return fail(HB_ERR_WORKSPACE, "plan was made for a different batch geometry");
    if (batch->total_q == 0) return ok();
    if (!(softmax_scale > 0.f) && !(softmax_scale <= 0.f))
      return fail(HB_ERR_INVALID_ARG, "softmax_scale is NaN");
    if ((s = check_ptr(q, "q")) != HB_OK) return s;
    if ((s = check_ptr(out, "out")) != HB_OK) return s;
    if ((s = check_ptr(k_cache, "k_cache")) != HB_OK) return s;
    if ((s = check_ptr(v_cache, "v_cache")) != HB_OK) return s;
    if (k_new && (s = check_ptr(k_new, "k_new")) != HB_OK) return s;
    if (v_new && (s = check_ptr(v_new, "v_new")) != HB_OK) return s;
    if (!d_workspace || (reinterpret_cast<uintptr_t>(d_workspace) & 255u))
      return fail(HB_ERR_INVALID_ARG, "d_workspace must be non-NULL and 256-byte aligned");
    DevState* dev = nullptr;
    if ((s = device_state(&dev)) != HB_OK) return s;
    if ((s = get_encoder()) != HB_OK) return s;

    const int Hq = batch->num_q_heads, Hkv = batch->num_kv_heads, D = batch->head_dim;
    const int g = Hq / Hkv;
    const float scale_log2 = softmax_scale * 1.4426950408889634f;
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // one launch: decode CTAs first, then one CTA per chunk item
    CUtensorMap dec_k, dec_v, chunk_q, chunk_k, chunk_v, chunk_knew, chunk_vnew;
    std::memset(&chunk_knew, 0, sizeof(chunk_knew));
    std::memset(&chunk_vnew, 0, sizeof(chunk_vnew));
    std::memset(&chunk_k, 0, sizeof(chunk_k));
    std::memset(&chunk_v, 0, sizeof(chunk_v));
    std::memset(&dec_k, 0, sizeof(dec_k));
    std::memset(&dec_v, 0, sizeof(dec_v));
    std::memset(&chunk_q, 0, sizeof(chunk_q));
    const int kvhb = h.decode_kvh_block;
    DecodeParams dp{};
    dp.group = g;
    dp.kvh_block = kvhb;
    if (h.num_decode_items > 0) {
      // pools viewed as [page][kv head][slot][head dim] boxes: dims are
      // (D, slot, kv head, page) with the pool's own strides
      const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPageSize, (cuuint64_t)Hkv,
                                  (cuuint64_t)batch->num_pages};
      const cuuint64_t strides[3] = {(cuuint64_t)Hkv * D * 2, (cuuint64_t)D * 2,
                                     (cuuint64_t)kPageSize * Hkv * D * 2};
      const cuuint32_t box[4] = {64, (cuuint32_t)kPageSize, (cuuint32_t)kvhb, 1};
      if ((s = encode_map(&dec_k, k_cache, 4, dims, strides, box, "decode K")) != HB_OK) return s;
      if ((s = encode_map(&dec_v, v_cache, 4, dims, strides, box, "decode V")) != HB_OK) return s;
      dp.items = reinterpret_cast<const DecodeItem*>(ws);
      dp.cta_offsets = reinterpret_cast<const int32_t*>(ws + h.ws_decode_offsets);
      dp.num_static = h.decode_grid;
      dp.num_dynamic = h.num_decode_dynamic;
      dp.num_items = h.num_decode_items;
      dp.counters = reinterpret_cast<int32_t*>(ws + h.ws_counters);
      dp.part_o = reinterpret_cast<float*>(ws + h.ws_partial_o);
      dp.part_ml = reinterpret_cast<float*>(ws + h.ws_partial_ml);
      dp.cu_q_len = batch->cu_q_len;
      dp.context_len = batch->context_len;
      dp.block_table = batch->block_table;
      dp.max_pages_per_seq = batch->max_pages_per_seq;
      dp.num_pages = batch->num_pages;
      dp.q = static_cast<const uint16_t*>(q);
      dp.out = static_cast<uint16_t*>(out);
      dp.num_q_heads = Hq;
      dp.num_kv_heads = Hkv;
      dp.scale_log2 = scale_log2;
      dp.dev_error = dev->err;
      dp.window = batch->sliding_window;
    }
    ChunkParams cp{};
    cp.group = g;
    if (h.num_chunk_items > 0) {
      const int tpt = h.chunk_tokens_per_tile;
      const cuuint64_t qdims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)batch->total_q};
      const cuuint64_t qstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
      const cuuint32_t qbox[3] = {64, (cuuint32_t)g, (cuuint32_t)tpt};
      if ((s = encode_map(&chunk_q, q, 3, qdims, qstr, qbox, "chunk Q")) != HB_OK) return s;
      // pools viewed as (D, kv head, token slot) with one box per page
      const cuuint64_t kdims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv,
                                   (cuuint64_t)batch->num_pages * kPageSize};
      const cuuint64_t kstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2};
      const cuuint32_t kbox[3] = {64, 1, (cuuint32_t)kPageSize};
      if ((s = encode_map(&chunk_k, k_cache, 3, kdims, kstr, kbox, "chunk K")) != HB_OK) return s;
      if ((s = encode_map(&chunk_v, v_cache, 3, kdims, kstr, kbox, "chunk V")) != HB_OK) return s;
      if (k_new && v_new) {
        // the new rows [total_q, Hkv, D] viewed as (D, kv head, token), the
        // same 16-token boxes as a page
        const cuuint64_t ndims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)batch->total_q};
        if ((s = encode_map(&chunk_knew, k_new, 3, ndims, kstr, kbox, "chunk K (new rows)")) != HB_OK)
          return s;
        if ((s = encode_map(&chunk_vnew, v_new, 3, ndims, kstr, kbox, "chunk V (new rows)")) != HB_OK)
          return s;
        cp.has_new = 1;
      } else {
        chunk_knew = chunk_k;
        chunk_vnew = chunk_v;
      }
      cp.items = reinterpret_cast<const ChunkItem*>(ws + (size_t)h.num_decode_items * sizeof(DecodeItem));
      cp.num_items = h.num_chunk_items;
      cp.cu_q_len = batch->cu_q_len;
      cp.context_len = batch->context_len;
      cp.block_table = batch->block_table;
      cp.max_pages_per_seq = batch->max_pages_per_seq;
      cp.num_pages = batch->num_pages;
      cp.out = static_cast<uint16_t*>(out);
      cp.num_q_heads = Hq;
      cp.num_kv_heads = Hkv;
      cp.tokens_per_tile = tpt;
      cp.scale_log2 = scale_log2;
      cp.dev_error = dev->err;
      cp.window = batch->sliding_window;
      cp.counters = reinterpret_cast<int32_t*>(ws + h.ws_chunk_counters);
      cp.part_o = reinterpret_cast<float*>(ws + h.ws_chunk_o);
      cp.part_ml = reinterpret_cast<float*>(ws + h.ws_chunk_ml);
    }
    if (h.num_decode_items > 0 || h.num_chunk_items > 0) {
      const bool early = follows_own_append(stream, batch, k_cache, v_cache);
      LaunchTimer t(1, st);
      cudaError_t e = launch_attention(dp, h.decode_grid, cp, D, dec_k, dec_v, chunk_q, chunk_k,
                                       chunk_v, chunk_knew, chunk_vnew, k_cache, v_cache, st,
                                       early, h.chunk_pairs_only);
      t.done();
      if (e != cudaSuccess) return cuda_fail(e, "attention launch");
      note_launch(stream, LastLaunch{});
      g_launches.fetch_add(1);
    }
    return ok();
  } catch (...) {
    return fail(HB_ERR_CUDA, "unexpected exception in hb_attention");
  }
}

extern "C" {

hb_status hb_check(void* stream) {
  try {
    DevState* dev = nullptr;
    hb_status s = device_state(&dev);
    if (s != HB_OK) return s;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int v = 0;
    e = cudaMemcpy(&v, dev->err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (v == 0) return ok();
    const int zero = 0;
    cudaMemcpy(dev->err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (v & HB_DEVERR_INDEX)
      return fail(HB_ERR_DEVICE_INDEX, "a kernel met a page index outside [0, num_pages) (word %d)", v);
    return fail(HB_ERR_TIMEOUT, "a kernel wait gave up (word %d)", v);
  } catch (...) {
    return fail(HB_ERR_CUDA, "unexpected exception in hb_check");
  }
}

hb_status hb_selftest_wait_timeout(void* stream) {
  try {
    DevState* dev = nullptr;
    hb_status s = device_state(&dev);
    if (s != HB_OK) return s;
    cudaError_t e = launch_wait_timeout(dev->err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    g_launches.fetch_add(1);
    return ok();
  } catch (...) {
    return fail(HB_ERR_CUDA, "unexpected exception in hb_selftest_wait_timeout");
  }
}

hb_status hb_selftest_flag_timeout(void* stream) {
  try {
    DevState* dev = nullptr;
    hb_status s = device_state(&dev);
    if (s != HB_OK) return s;
    cudaError_t e = launch_flag_timeout(dev->err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    g_launches.fetch_add(1);
    return ok();
  } catch (...) {
    return fail(HB_ERR_CUDA, "unexpected exception in hb_selftest_flag_timeout");
  }
}

hb_status hb_timing_enable(int32_t enable) {
  if (enable < 0 || enable > 2) return fail(HB_ERR_INVALID_ARG, "timing mode must be 0, 1 or 2");
  std::lock_guard<std::mutex> lk(g_time_mu);
  if (enable == 1) {
    for (auto& r : g_recs) {
      g_event_pool.push_back(r.a);
      g_event_pool.push_back(r.b);
    }
    g_recs.clear();
  }
  g_timing = enable != 0;
  return ok();
}

hb_status hb_timing_read(double* total_ms, int32_t* launches) {
  if (!total_ms || !launches) return fail(HB_ERR_INVALID_ARG, "NULL output");
  std::lock_guard<std::mutex> lk(g_time_mu);
  for (int k = 0; k < HB_NUM_KERNEL_IDS; ++k) {
    total_ms[k] = 0.0;
    launches[k] = 0;
  }
  for (auto& r : g_recs) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, r.a, r.b);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    if (r.kernel >= 0 && r.kernel < HB_NUM_KERNEL_IDS) {
      total_ms[r.kernel] += ms;
      launches[r.kernel] += 1;
    }
  }
  return ok();
}

hb_status hb_timing_durations(int32_t kernel, float* ms, int32_t max, int32_t* n) {
  if (!n || (max > 0 && !ms)) return fail(HB_ERR_INVALID_ARG, "NULL output");
  if (kernel < 0 || kernel >= HB_NUM_KERNEL_IDS)
    return fail(HB_ERR_INVALID_ARG, "kernel id %d", kernel);
  std::lock_guard<std::mutex> lk(g_time_mu);
  int32_t k = 0;
  for (auto& r : g_recs) {
    if (r.kernel != kernel) continue;
    if (k < max) {
      cudaError_t e = cudaEventSynchronize(r.b);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
      e = cudaEventElapsedTime(&ms[k], r.a, r.b);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
    }
    ++k;
  }
  *n = k;
  return ok();
}

int64_t hb_launch_count(void) { return g_launches.load(); }

}  // extern "C"
