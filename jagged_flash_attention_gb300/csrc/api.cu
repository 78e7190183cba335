// Host side of the C ABI declared in include/jfa.h: argument validation,
// stream-ordered scratch memory, TMA tensor-map encoding and the launch
// sequence of the forward and backward passes.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "jfa.h"

namespace jfa {
// Device error word, OR-ed by the kernels (bits in ptx.cuh).
__device__ int g_device_error;
}  // namespace jfa

namespace {

// Largest head count: work items hold (head << 16) | tile in an int32.
constexpr int kMaxHeads = 32767;

using namespace jfa;

thread_local std::string t_last_error;

// Kernel launch accounting: a process-wide count of enqueued kernels and,
// while profiling is on, a CUDA event pair around every launch, recorded on
// the launch's own stream (read back by jfa_profile_read).
std::atomic<long long> g_launch_count{0};
std::atomic<int> g_profile_on{0};
std::atomic<unsigned> g_profile_kinds{~0u};  // bit k: record kind k
struct ProfRecord {
  int kind;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
std::vector<ProfRecord> g_prof;

template <class F>
cudaError_t run_kernel(jfa_kernel_kind kind, cudaStream_t stream, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  const bool prof = g_profile_on.load(std::memory_order_relaxed) != 0 &&
                    ((g_profile_kinds.load(std::memory_order_relaxed) >> kind) & 1u) != 0 &&
                    cudaEventCreate(&a) == cudaSuccess && cudaEventCreate(&b) == cudaSuccess;
  if (prof) cudaEventRecord(a, stream);
  const cudaError_t e = launch();
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  if (prof) {
    cudaEventRecord(b, stream);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back({static_cast<int>(kind), a, b});
  } else {
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
  }
  return e;
}

jfa_status fail(jfa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  cudaMemPool_t pool = nullptr;
  int* err = nullptr;  // device address of g_device_error
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool validate_mode() {
  static const bool v = [] {
    const char* e = std::getenv("JFA_VALIDATE");
    return e && e[0] == '1';
  }();
  return v;
}

jfa_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(JFA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(JFA_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess)
      return fail(JFA_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
    s.sms = prop.multiProcessorCount;
    s.cc_major = prop.major;
    s.cc_minor = prop.minor;
    if (!(prop.major == 10 && prop.minor == 3))
      return fail(JFA_ERR_UNSUPPORTED, "device %s is sm_%d%d; this library is built for sm_103a",
                  prop.name, prop.major, prop.minor);
    cudaMemPoolProps pp;
    memset(&pp, 0, sizeof(pp));
    pp.allocType = cudaMemAllocationTypePinned;
    pp.location.type = cudaMemLocationTypeDevice;
    pp.location.id = dev;
    e = cudaMemPoolCreate(&s.pool, &pp);
    if (e != cudaSuccess) return fail(JFA_ERR_CUDA, "cudaMemPoolCreate: %s", cudaGetErrorString(e));
    uint64_t keep = UINT64_MAX;  // keep freed scratch in the pool between calls
    cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_device_error);
    if (e != cudaSuccess)
      return fail(JFA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || !fn || q != cudaDriverEntryPointSuccess)
        return fail(JFA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.ready = true;
  }
  *out = &s;
  return JFA_OK;
}

// [rows, H, D] bf16 tensor viewed as a 3-D map (D, H, rows), box 64 x 1 x
// box_rows (128 by default), 128-byte swizzle: one TMA copy of 128 rows
// fills one 16 KB swizzle-atom slab.
jfa_status map_rows(CUtensorMap* m, const void* ptr, int D, int H, long long rows, const char* nm,
                    unsigned box_rows = 128) {
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(JFA_ERR_CUDA, "tensor map for %s failed (%d)", nm, (int)r);
  return JFA_OK;
}

// [B, Lq, H, D] bf16 tensor as a 4-D map (D, H, Lq, B), box 64 x 1 x box_rows x 1.
jfa_status map_bq(CUtensorMap* m, const void* ptr, int D, int H, int Lq, int B, const char* nm,
                  unsigned box_rows = 128) {
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)Lq, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)Lq * H * D * 2};
  cuuint32_t box[4] = {64, 1, box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(JFA_ERR_CUDA, "tensor map for %s failed (%d)", nm, (int)r);
  return JFA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long cdivll(long long a, long long b) { return (a + b - 1) / b; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Shape {
  int B, H, D, max_len, Lq, broadcast, causal;
  int Hkv, G;       // K/V heads; query heads per K/V head (GQA)
  int wl, wr;       // window bounds as given (-1: unbounded)
  int kwl, kwr;     // the kernels' bounds: kNoWindow when unbounded, causal: kwr = 0
  int local;        // a local mask: causal or a window
  float scale;
  long long Tcap;  // upper bound of T used to size scratch and tensor maps
};

// dK/dV pass on pairs of CTAs (cta_group::2 products over two key blocks):
// JFA_KV_PAIR=1 selects it where it applies (D = 128, no local mask; for
// broadcast-Q, the two-pass backward); read on every call.
bool kv_pair_mode(const Shape& s) {
  const char* e = std::getenv("JFA_KV_PAIR");
  return e != nullptr && e[0] == '1' && s.D == 128 && !s.local;
}

// GQA group and local mask of a kernel parameter block.
template <class P>
void set_variant(P& p, const Shape& s) {
  p.G = s.G;
  p.wl = s.kwl;
  p.wr = s.kwr;
}

jfa_status check_common(const Shape& s, const void* q, const void* k, const void* v,
                        const int32_t* offsets) {
  if (s.B < 1) return fail(JFA_ERR_INVALID_ARG, "B must be >= 1 (got %d)", s.B);
  // Work items carry the head in bits 16-30 of a signed 32-bit word.
  if (s.H < 1 || s.H > kMaxHeads)
    return fail(JFA_ERR_INVALID_ARG, "H must be in [1, %d] (got %d)", kMaxHeads, s.H);
  if (s.D != 64 && s.D != 128) return fail(JFA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", s.D);
  if (s.max_len < 0) return fail(JFA_ERR_INVALID_ARG, "max_len must be >= 0");
  if (cdivll(s.max_len, kBN) > 65535 || cdivll(s.Lq, kBM) > 65535)
    return fail(JFA_ERR_INVALID_ARG, "sequence length too large");
  if ((long long)s.B * s.max_len >= (1LL << 31))
    return fail(JFA_ERR_INVALID_ARG, "B * max_len must be < 2^31");
  if (!std::isfinite(s.scale) || !(s.scale > 0.f))
    return fail(JFA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (s.Hkv < 1 || s.Hkv > s.H || s.H % s.Hkv != 0)
    return fail(JFA_ERR_INVALID_ARG, "H_kv must divide H (got H = %d, H_kv = %d)", s.H, s.Hkv);
  if (s.wl < -1 || s.wr < -1)
    return fail(JFA_ERR_INVALID_ARG, "window bounds must be >= -1 (-1: unbounded)");
  if (s.causal && s.wr > 0)
    return fail(JFA_ERR_INVALID_ARG, "causal masking bounds the window's right side by 0 (got %d)",
                s.wr);
  if (s.broadcast && s.causal)
    return fail(JFA_ERR_UNSUPPORTED, "causal masking is supported for self-attention only");
  if (s.broadcast && (s.wl >= 0 || s.wr >= 0))
    return fail(JFA_ERR_UNSUPPORTED, "sliding windows are supported for self-attention only");
  if (s.broadcast && s.Lq < 1) return fail(JFA_ERR_INVALID_ARG, "q_len must be >= 1 in broadcast mode");
  if (!offsets || (reinterpret_cast<uintptr_t>(offsets) & 3u))
    return fail(JFA_ERR_INVALID_ARG, "offsets must be a non-null, 4-byte aligned device pointer");
  if (!q || !k || !v) return fail(JFA_ERR_INVALID_ARG, "q, k, v must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v))
    return fail(JFA_ERR_INVALID_ARG, "q, k, v must be 16-byte aligned");
  return JFA_OK;
}

jfa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(JFA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

jfa_status sync_and_read_error_word(cudaStream_t stream);

// With JFA_VALIDATE=1 every entry point synchronises its stream and reports
// device-side errors before returning.
jfa_status finish(cudaStream_t stream) {
  if (!validate_mode()) return JFA_OK;
  return sync_and_read_error_word(stream);
}

// Broadcast-Q forward with a short dense Q (one 128-row tile): the key
// tiles of all sequences cut into equal chunks per head (the dQ-pass chunk
// list), a streamed forward over the chunks, and the merge of the sequences
// that a chunk boundary splits.
jfa_status do_fwd_bs(DeviceState* ds, const Shape& s, const void* q, const void* k, const void* v,
                     const int32_t* offsets, void* out, float* lse, cudaStream_t stream) {
  jfa_status st;
  const long long chunk_cap = std::max<long long>(1, cdivll(2LL * ds->sms, s.H));
  const long long cap = chunk_cap * s.H;
  size_t off = 256;
  const size_t items_off = off;
  off = align256(off + cap * sizeof(QbItem));
  const size_t ktoff_off = off;
  off = align256(off + (s.B + 1) * sizeof(int));
  const size_t parto_off = off;
  off = align256(off + (size_t)cap * 2 * kBM * s.D * sizeof(float));
  const size_t partl_off = off;
  off = align256(off + (size_t)cap * 2 * kBM * sizeof(float));
  CUtensorMap tq, tk, tv;
  // a dense Q of at most 64 rows is loaded in 16-row boxes (the spread layout)
  if ((st = map_rows(&tq, q, s.D, s.H, s.Lq, "q", fwd_bs_spread(s.Lq) ? 16 : 128)) != JFA_OK)
    return st;
  if ((st = map_rows(&tk, k, s.D, s.Hkv, s.Tcap, "k")) != JFA_OK) return st;
  if ((st = map_rows(&tv, v, s.D, s.Hkv, s.Tcap, "v")) != JFA_OK) return st;
  void* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, off, ds->pool, stream);
  if (e != cudaSuccess) return fail(JFA_ERR_WORKSPACE, "scratch allocation: %s", cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  WorkHeader* hdr = reinterpret_cast<WorkHeader*>(base);
  QbItem* items = reinterpret_cast<QbItem*>(base + items_off);
  int* kt_off = reinterpret_cast<int*>(base + ktoff_off);
  QbSchedParams qp{offsets, s.B, s.H, s.Lq, s.max_len, (int)chunk_cap, kt_off, items, (int)cap,
                   hdr, ds->err};
  e = run_kernel(JFA_KERNEL_SCHED, stream, [&] { return launch_qb_sched(qp, stream); });
  FwdParams fp;
  memset(&fp, 0, sizeof(fp));
  fp.offsets = offsets;
  fp.B = s.B;
  fp.H = s.H;
  fp.Lq = s.Lq;
  fp.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
  fp.out = static_cast<__nv_bfloat16*>(out);
  fp.lse = lse;
  fp.hdr = hdr;
  fp.err = ds->err;
  fp.qb_items = items;
  fp.kt_off = kt_off;
  fp.part_o = reinterpret_cast<float*>(base + parto_off);
  fp.part_lse = reinterpret_cast<float*>(base + partl_off);
  set_variant(fp, s);
  if (e == cudaSuccess)
    e = run_kernel(JFA_KERNEL_FWD, stream, [&] {
      return launch_fwd_bs(s.D, tq, tk, tv, fp, (int)std::min<long long>(ds->sms, cap), stream);
    });
  if (e == cudaSuccess)
    e = run_kernel(JFA_KERNEL_FWD_COMBINE, stream,
                   [&] { return launch_fwd_combine(s.D, fp, ds->sms, stream); });
  cudaError_t e2 = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch free");
  return finish(stream);
}

jfa_status do_fwd(const Shape& s, const void* q, const void* k, const void* v,
                  const int32_t* offsets, void* out, float* lse, cudaStream_t stream) {
  jfa_status st = check_common(s, q, k, v, offsets);
  if (st != JFA_OK) return st;
  if (!out || !aligned16(out)) return fail(JFA_ERR_INVALID_ARG, "out must be non-null, 16-byte aligned");
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(JFA_ERR_INVALID_ARG, "lse must be non-null, 4-byte aligned");
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != JFA_OK) return st;
  cudaError_t e;
  if (s.max_len == 0) {  // every sequence is empty
    if (s.broadcast) {
      e = run_kernel(JFA_KERNEL_FILL, stream, [&] {
        return launch_fill_empty(
            static_cast<__nv_bfloat16*>(out), lse, (long long)s.B * s.Lq * s.H, s.D, stream);
      });
      if (e != cudaSuccess) return cuda_fail(e, "fill launch");
    }
    return finish(stream);
  }
  if (s.broadcast && fwd_bs_supported(s.Lq)) return do_fwd_bs(ds, s, q, k, v, offsets, out, lse, stream);
  const long long qt = s.broadcast ? cdivll(s.Lq, kFwdRows) : cdivll(s.max_len, kFwdRows);
  const long long cap = (long long)s.H * s.B * qt;
  if (cap >= (1LL << 31)) return fail(JFA_ERR_INVALID_ARG, "work list too large");
  const size_t items_off = 256;
  const size_t bytes = align256(items_off + cap * sizeof(Item));
  CUtensorMap tq, tk, tv;
  if ((st = map_rows(&tq, q, s.D, s.H, s.broadcast ? s.Lq : s.Tcap, "q")) != JFA_OK) return st;
  if ((st = map_rows(&tk, k, s.D, s.Hkv, s.Tcap, "k")) != JFA_OK) return st;
  if ((st = map_rows(&tv, v, s.D, s.Hkv, s.Tcap, "v")) != JFA_OK) return st;
  void* scratch = nullptr;
  e = cudaMallocFromPoolAsync(&scratch, bytes, ds->pool, stream);
  if (e != cudaSuccess) return fail(JFA_ERR_WORKSPACE, "scratch allocation: %s", cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  WorkHeader* hdr = reinterpret_cast<WorkHeader*>(base);
  Item* items = reinterpret_cast<Item*>(base + items_off);
  SchedParams sp{offsets, s.B, s.H, s.Lq, s.max_len, s.local, s.broadcast, 0, kFwdRows,
                 items, (int)cap, hdr, ds->err, s.kwl, s.kwr};
  e = run_kernel(JFA_KERNEL_SCHED, stream, [&] {
    return launch_sched(sp, stream);
  });
  if (e == cudaSuccess) {
    FwdParams fp;
    memset(&fp, 0, sizeof(fp));
    set_variant(fp, s);
    fp.offsets = offsets;
    fp.B = s.B;
    fp.H = s.H;
    fp.Lq = s.Lq;
    fp.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.lse = lse;
    fp.items = items;
    fp.hdr = hdr;
    fp.err = ds->err;
    // One CTA per possible item: the forward takes work by cancelling CTAs
    // that have not started (cluster launch control).
    const int grid = (int)cap;
    e = run_kernel(JFA_KERNEL_FWD, stream, [&] {
      return launch_fwd(s.D, s.local, s.broadcast, tq, tk, tv, fp, grid, stream);
    });
  }
  cudaError_t e2 = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch free");
  return finish(stream);
}

// Self-attention backward: dK/dV pass (K/V-block outer) and dQ pass
// (query-tile outer, dQ accumulated on chip), so no fp32 dQ accumulator is
// needed.  Work lists, Delta and the two headers are the only scratch.
jfa_status do_bwd_self(DeviceState* ds, const Shape& s, const void* q, const void* k,
                       const void* v, const int32_t* offsets, const void* out, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, cudaStream_t stream) {
  jfa_status st;
  const long long cap_kv = (long long)s.Hkv * s.B * cdivll(s.max_len, kBN);
  const long long cap_q = (long long)s.H * s.B * cdivll(s.max_len, kFwdRows);
  if (cap_kv >= (1LL << 31) || cap_q >= (1LL << 31))
    return fail(JFA_ERR_INVALID_ARG, "work list too large");
  const long long stat_stride = stat_copy_floats((long long)s.H * s.Tcap);
  size_t off = 0;
  const size_t hkv_off = off;
  off = align256(off + 256 + cap_kv * sizeof(Item));
  const size_t hq_off = off;
  off = align256(off + 256 + cap_q * sizeof(Item));
  const size_t stat_off = off;
  off = align256(off + kStatCopies * stat_stride * sizeof(float));
  CUtensorMap tq, tk, tv, tdo;
  if ((st = map_rows(&tq, q, s.D, s.H, s.Tcap, "q")) != JFA_OK) return st;
  if ((st = map_rows(&tk, k, s.D, s.Hkv, s.Tcap, "k")) != JFA_OK) return st;
  if ((st = map_rows(&tv, v, s.D, s.Hkv, s.Tcap, "v")) != JFA_OK) return st;
  if ((st = map_rows(&tdo, dout, s.D, s.H, s.Tcap, "dout")) != JFA_OK) return st;
  CUtensorMap tdk, tdv;
  if ((st = map_rows(&tdk, dk, s.D, s.Hkv, s.Tcap, "dk")) != JFA_OK) return st;
  if ((st = map_rows(&tdv, dv, s.D, s.Hkv, s.Tcap, "dv")) != JFA_OK) return st;
  // the pair variant also reads half-tiles of Q and dO (64-row boxes)
  const bool pair = kv_pair_mode(s);
  CUtensorMap tq_h, tdo_h;
  if (pair) {
    if ((st = map_rows(&tq_h, q, s.D, s.H, s.Tcap, "q", 64)) != JFA_OK) return st;
    if ((st = map_rows(&tdo_h, dout, s.D, s.H, s.Tcap, "dout", 64)) != JFA_OK) return st;
  }
  void* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, off, ds->pool, stream);
  if (e != cudaSuccess) return fail(JFA_ERR_WORKSPACE, "scratch allocation: %s", cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  WorkHeader* hdr_kv = reinterpret_cast<WorkHeader*>(base + hkv_off);
  Item* items_kv = reinterpret_cast<Item*>(base + hkv_off + 256);
  WorkHeader* hdr_q = reinterpret_cast<WorkHeader*>(base + hq_off);
  Item* items_q = reinterpret_cast<Item*>(base + hq_off + 256);
  float* stat = reinterpret_cast<float*>(base + stat_off);
  // dK/dV items over the K/V heads, dQ items over the query heads
  SchedParams sk{offsets, s.B, s.Hkv, s.Lq, s.max_len, s.local, 0, 1, kBM,
                 items_kv, (int)cap_kv, hdr_kv, ds->err, s.kwl, s.kwr};
  sk.kpair = pair ? 2 : 1;
  SchedParams sq{offsets, s.B, s.H, s.Lq, s.max_len, s.local, 0, 0, kFwdRows,
                 items_q, (int)cap_q, hdr_q, ds->err, s.kwl, s.kwr};
  BwdParams bp;
  memset(&bp, 0, sizeof(bp));
  set_variant(bp, s);
  bp.Hkv = s.Hkv;
  bp.offsets = offsets;
  bp.B = s.B;
  bp.H = s.H;
  bp.Lq = 0;
  bp.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
  bp.scale = s.scale;
  bp.lse = lse;
  bp.stat = stat;
  bp.stat_stride = stat_stride;
  bp.dq = static_cast<__nv_bfloat16*>(dq);
  bp.dk = static_cast<__nv_bfloat16*>(dk);
  bp.dv = static_cast<__nv_bfloat16*>(dv);
  bp.err = ds->err;
  {
    // One launch: both work lists and the row statistics.
    PrepParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.out = static_cast<const __nv_bfloat16*>(out);
    pp.dout = static_cast<const __nv_bfloat16*>(dout);
    pp.offsets = offsets;
    pp.lse = lse;
    pp.stat = stat;
    pp.stat_stride = stat_stride;
    pp.Tcap = s.Tcap;
    pp.B = s.B;
    pp.H = s.H;
    pp.D = s.D;
    pp.n_sched = 2;
    pp.sched[0] = sk;
    pp.sched[1] = sq;
    e = run_kernel(JFA_KERNEL_PREP, stream, [&] {
      return launch_bwd_prep(pp, ds->sms, stream);
    });
  }
  if (e == cudaSuccess) {
    bp.items = items_kv;
    bp.hdr = hdr_kv;
    e = run_kernel(pair ? JFA_KERNEL_BWD_KV_PAIR : JFA_KERNEL_BWD_KV, stream, [&] {
      return launch_bwd_kv(s.D, s.local, false, tq, tk, tv, tdo, tdk, tdv, bp,
                           (int)std::min<long long>(ds->sms, pair ? 2 * cap_kv : cap_kv), stream,
                           pair ? &tq_h : nullptr, pair ? &tdo_h : nullptr);
    });
  }
  if (e == cudaSuccess) {
    bp.items = items_q;
    bp.hdr = hdr_q;
    e = run_kernel(JFA_KERNEL_BWD_Q, stream, [&] {
      return launch_bwd_q(
          s.D, s.local, tq, tk, tv, tdo, bp, (int)std::min<long long>(ds->sms, cap_q), stream);
    });
  }
  cudaError_t e2 = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch free");
  return finish(stream);
}

// Broadcast-Q backward, two passes like self-attention: a dK/dV pass whose
// query tiles are the dense Q's (items: sequence, head, key block), and a dQ
// pass over equal chunks of the key-tile stream of all sequences (items:
// chunk, head, query-tile pair) that keeps dQ in tensor memory and writes
// one fp32 partial per item; a finalize kernel sums the partials in chunk
// order.  Scratch: the two work lists, key-tile prefix per sequence, the row
// statistics (padded to whole query tiles) and the partials.
jfa_status do_bwd_bcast(DeviceState* ds, const Shape& s, const void* q, const void* k,
                        const void* v, const int32_t* offsets, const void* out, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, cudaStream_t stream) {
  jfa_status st;
  const long long cap_kv = (long long)s.Hkv * s.B * cdivll(s.max_len, kBN);
  const long long pairs = cdivll(s.Lq, kQbRows);
  // chunks per (head, pair): about two items per SM in all
  const long long chunk_cap = std::max<long long>(1, cdivll(2LL * ds->sms, s.H * pairs));
  const long long cap_qb = chunk_cap * s.H * pairs;
  const long long lq_pad = cdivll(s.Lq, kBM) * kBM;
  if (cap_kv >= (1LL << 31) || (long long)s.B * s.H * lq_pad >= (1LL << 40))
    return fail(JFA_ERR_INVALID_ARG, "work list too large");
  // A short dense Q (one tile, D = 64): dK, dV and dQ in one pass over K / V
  // (one query head per K/V head: with GQA, dK / dV sum over several query
  // heads, which the two-pass path does in its dK/dV pass).
  const bool one_pass = bwd_bs_supported(s.D, s.Lq) && s.G == 1;
  size_t off = 0;
  const size_t hkv_off = off;
  off = align256(off + 256 + (one_pass ? 0 : cap_kv) * sizeof(Item));
  const size_t hqb_off = off;
  off = align256(off + 256 + cap_qb * sizeof(QbItem));
  const size_t ktoff_off = off;
  off = align256(off + (s.B + 1) * sizeof(int));
  const size_t stat_off = off;
  off = align256(off + 2 * (size_t)s.B * s.H * lq_pad * sizeof(float));
  const size_t part_off = off;
  off = align256(off + (size_t)cap_qb * 2 * kBM * s.D * sizeof(float));
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if ((st = map_rows(&tq, q, s.D, s.H, s.Lq, "q")) != JFA_OK) return st;
  if ((st = map_rows(&tk, k, s.D, s.Hkv, s.Tcap, "k")) != JFA_OK) return st;
  if ((st = map_rows(&tv, v, s.D, s.Hkv, s.Tcap, "v")) != JFA_OK) return st;
  if ((st = map_bq(&tdo, dout, s.D, s.H, s.Lq, s.B, "dout")) != JFA_OK) return st;
  if ((st = map_rows(&tdk, dk, s.D, s.Hkv, s.Tcap, "dk")) != JFA_OK) return st;
  if ((st = map_rows(&tdv, dv, s.D, s.Hkv, s.Tcap, "dv")) != JFA_OK) return st;
  const bool pair = !one_pass && kv_pair_mode(s);
  CUtensorMap tq_h, tdo_h;
  if (pair) {
    if ((st = map_rows(&tq_h, q, s.D, s.H, s.Lq, "q", 64)) != JFA_OK) return st;
    if ((st = map_bq(&tdo_h, dout, s.D, s.H, s.Lq, s.B, "dout", 64)) != JFA_OK) return st;
  }
  void* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, off, ds->pool, stream);
  if (e != cudaSuccess) return fail(JFA_ERR_WORKSPACE, "scratch allocation: %s", cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  WorkHeader* hdr_kv = reinterpret_cast<WorkHeader*>(base + hkv_off);
  Item* items_kv = reinterpret_cast<Item*>(base + hkv_off + 256);
  WorkHeader* hdr_qb = reinterpret_cast<WorkHeader*>(base + hqb_off);
  QbItem* items_qb = reinterpret_cast<QbItem*>(base + hqb_off + 256);
  int* kt_off = reinterpret_cast<int*>(base + ktoff_off);
  float* stat = reinterpret_cast<float*>(base + stat_off);
  float* part = reinterpret_cast<float*>(base + part_off);
  {
    PrepParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.out = static_cast<const __nv_bfloat16*>(out);
    pp.dout = static_cast<const __nv_bfloat16*>(dout);
    pp.offsets = offsets;
    pp.lse = lse;
    pp.stat = stat;
    pp.B = s.B;
    pp.H = s.H;
    pp.D = s.D;
    pp.Lq = s.Lq;
    pp.broadcast = 1;
    pp.n_sched = one_pass ? 1 : 2;
    pp.qb_only = one_pass ? 1 : 0;
    pp.sched[0] = SchedParams{offsets, s.B, s.Hkv, s.Lq, s.max_len, 0, 1, 1, kBM,
                              items_kv, (int)cap_kv, hdr_kv, ds->err};
    pp.sched[0].kpair = pair ? 2 : 1;
    pp.qb = QbSchedParams{offsets, s.B, s.H, s.Lq, s.max_len, (int)chunk_cap, kt_off,
                          items_qb, (int)cap_qb, hdr_qb, ds->err};
    e = run_kernel(JFA_KERNEL_PREP, stream, [&] {
      return launch_bwd_prep(pp, ds->sms, stream);
    });
  }
  BwdParams bp;
  memset(&bp, 0, sizeof(bp));
  set_variant(bp, s);
  bp.Hkv = s.Hkv;
  bp.offsets = offsets;
  bp.B = s.B;
  bp.H = s.H;
  bp.Lq = s.Lq;
  bp.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
  bp.scale = s.scale;
  bp.lse = lse;
  bp.stat = stat;
  bp.dq_part = part;
  bp.dk = static_cast<__nv_bfloat16*>(dk);
  bp.dv = static_cast<__nv_bfloat16*>(dv);
  bp.err = ds->err;
  if (e == cudaSuccess && one_pass) {
    bp.qb_items = items_qb;
    bp.hdr = hdr_qb;
    e = run_kernel(JFA_KERNEL_BWD_BCAST_ONEPASS, stream, [&] {
      return launch_bwd_bs(tq, tk, tv, tdo, bp, (int)std::min<long long>(ds->sms, cap_qb), stream);
    });
  }
  if (e == cudaSuccess && !one_pass) {
    bp.items = items_kv;
    bp.hdr = hdr_kv;
    e = run_kernel(pair ? JFA_KERNEL_BWD_KV_PAIR : JFA_KERNEL_BWD_KV, stream, [&] {
      return launch_bwd_kv(s.D, false, true, tq, tk, tv, tdo, tdk, tdv, bp,
                           (int)std::min<long long>(ds->sms, pair ? 2 * cap_kv : cap_kv), stream,
                           pair ? &tq_h : nullptr, pair ? &tdo_h : nullptr);
    });
  }
  if (e == cudaSuccess && !one_pass) {
    bp.items = nullptr;
    bp.qb_items = items_qb;
    bp.hdr = hdr_qb;
    e = run_kernel(JFA_KERNEL_BWD_Q_BCAST, stream, [&] {
      return launch_bwd_qb(s.D, tq, tk, tv, tdo, bp, (int)std::min<long long>(ds->sms, cap_qb),
                           stream);
    });
  }
  if (e == cudaSuccess) {
    FinParams fp;
    fp.part = part;
    fp.dq = static_cast<__nv_bfloat16*>(dq);
    fp.scale = s.scale;
    fp.H = s.H;
    fp.D = s.D;
    fp.Lq = s.Lq;
    fp.hdr = hdr_qb;
    e = run_kernel(JFA_KERNEL_FINALIZE, stream, [&] {
      return launch_finalize(fp, ds->sms, stream);
    });
  }
  cudaError_t e2 = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch free");
  return finish(stream);
}

jfa_status do_bwd(const Shape& s, const void* q, const void* k, const void* v,
                  const int32_t* offsets, const void* out, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, cudaStream_t stream) {
  jfa_status st = check_common(s, q, k, v, offsets);
  if (st != JFA_OK) return st;
  if (!out || !dout || !dq || !dk || !dv)
    return fail(JFA_ERR_INVALID_ARG, "out, dout, dq, dk, dv must be non-null");
  if (!aligned16(out) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(JFA_ERR_INVALID_ARG, "out, dout, dq, dk, dv must be 16-byte aligned");
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(JFA_ERR_INVALID_ARG, "lse must be non-null, 4-byte aligned");
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != JFA_OK) return st;
  cudaError_t e;
  if (s.max_len == 0) {
    if (s.broadcast) {  // no keys anywhere: dq = 0
      e = run_kernel(JFA_KERNEL_FILL, stream, [&] {
        return launch_fill_empty(
            static_cast<__nv_bfloat16*>(dq), nullptr, (long long)s.Lq * s.H, s.D, stream);
      });
      if (e != cudaSuccess) return cuda_fail(e, "fill launch");
    }
    return finish(stream);
  }
  if (!s.broadcast)
    return do_bwd_self(ds, s, q, k, v, offsets, out, lse, dout, dq, dk, dv, stream);
  return do_bwd_bcast(ds, s, q, k, v, offsets, out, lse, dout, dq, dk, dv, stream);
}

Shape make_shape(int B, int H, int Hkv, int D, int max_len, int q_len, int broadcast_q,
                 int causal, int window_left, int window_right, float scale) {
  Shape s;
  s.B = B;
  s.H = H;
  s.Hkv = Hkv;
  s.G = (Hkv > 0 && H % Hkv == 0) ? H / Hkv : 1;
  s.D = D;
  s.max_len = max_len;
  s.Lq = broadcast_q ? q_len : 0;
  s.broadcast = broadcast_q ? 1 : 0;
  s.causal = causal ? 1 : 0;
  s.wl = window_left;
  s.wr = window_right;
  s.kwl = window_left >= 0 ? window_left : kNoWindow;
  s.kwr = s.causal ? 0 : (window_right >= 0 ? window_right : kNoWindow);
  s.local = (s.causal || window_left >= 0 || window_right >= 0) ? 1 : 0;
  s.scale = scale;
  s.Tcap = (long long)(B > 0 ? B : 0) * (max_len > 0 ? max_len : 0);
  return s;
}

}  // namespace

extern "C" {

jfa_status jfa_fwd(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                   int H, int D, int max_len, int broadcast_q, int causal, float scale, void* out,
                   float* lse, cudaStream_t stream) {
  if (broadcast_q)
    return fail(JFA_ERR_INVALID_ARG,
                "broadcast_q=1 needs the dense Q length: call jfa_fwd_bq with q_len");
  t_last_error.clear();
  return do_fwd(make_shape(B, H, H, D, max_len, 0, 0, causal, -1, -1, scale), q, k, v, offsets,
                out, lse, stream);
}

jfa_status jfa_bwd(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                   int H, int D, int max_len, int broadcast_q, int causal, float scale,
                   const void* out, const float* lse, const void* dout, void* dq, void* dk,
                   void* dv, cudaStream_t stream) {
  if (broadcast_q)
    return fail(JFA_ERR_INVALID_ARG,
                "broadcast_q=1 needs the dense Q length: call jfa_bwd_bq with q_len");
  t_last_error.clear();
  return do_bwd(make_shape(B, H, H, D, max_len, 0, 0, causal, -1, -1, scale), q, k, v, offsets,
                out, lse, dout, dq, dk, dv, stream);
}

jfa_status jfa_fwd_bq(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int D, int max_len, int q_len, int broadcast_q, int causal,
                      float scale, void* out, float* lse, cudaStream_t stream) {
  t_last_error.clear();
  return do_fwd(make_shape(B, H, H, D, max_len, q_len, broadcast_q, causal, -1, -1, scale), q, k,
                v, offsets, out, lse, stream);
}

jfa_status jfa_fwd_ex(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int H_kv, int D, int max_len, int q_len, int broadcast_q, int causal,
                      int window_left, int window_right, float scale, void* out, float* lse,
                      cudaStream_t stream) {
  t_last_error.clear();
  return do_fwd(make_shape(B, H, H_kv, D, max_len, q_len, broadcast_q, causal, window_left,
                           window_right, scale),
                q, k, v, offsets, out, lse, stream);
}

jfa_status jfa_bwd_bq(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int D, int max_len, int q_len, int broadcast_q, int causal,
                      float scale, const void* out, const float* lse, const void* dout, void* dq,
                      void* dk, void* dv, cudaStream_t stream) {
  t_last_error.clear();
  return do_bwd(make_shape(B, H, H, D, max_len, q_len, broadcast_q, causal, -1, -1, scale), q, k,
                v, offsets, out, lse, dout, dq, dk, dv, stream);
}

jfa_status jfa_bwd_ex(const void* q, const void* k, const void* v, const int32_t* offsets, int B,
                      int H, int H_kv, int D, int max_len, int q_len, int broadcast_q, int causal,
                      int window_left, int window_right, float scale, const void* out,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      cudaStream_t stream) {
  t_last_error.clear();
  return do_bwd(make_shape(B, H, H_kv, D, max_len, q_len, broadcast_q, causal, window_left,
                           window_right, scale),
                q, k, v, offsets, out, lse, dout, dq, dk, dv, stream);
}

jfa_status jfa_block_select(const void* q, const void* k, const int32_t* offsets, int B, int H,
                            int H_kv, int D, int max_len, int q_len, int broadcast_q,
                            int permille, int32_t* blocks, int32_t* counts, cudaStream_t stream) {
  return jfa_block_select_ex(q, k, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, 0, -1, -1,
                             permille, blocks, counts, stream);
}

jfa_status jfa_block_select_ex(const void* q, const void* k, const int32_t* offsets, int B, int H,
                               int H_kv, int D, int max_len, int q_len, int broadcast_q,
                               int causal, int window_left, int window_right, int permille,
                               int32_t* blocks, int32_t* counts, cudaStream_t stream) {
  t_last_error.clear();
  Shape s = make_shape(B, H, H_kv, D, max_len, q_len, broadcast_q, causal, window_left,
                       window_right, 1.f);
  jfa_status st = check_common(s, q, k, k, offsets);
  if (st != JFA_OK) return st;
  if (permille < 1 || permille > 1000)
    return fail(JFA_ERR_INVALID_ARG, "permille must be in [1, 1000] (got %d)", permille);
  if (B > 65535) return fail(JFA_ERR_INVALID_ARG, "block-sparse: B must be <= 65535");
  const long long kcap = cdivll(max_len, kBN), nqb = cdivll(s.broadcast ? s.Lq : max_len, kFwdRows);
  if (kcap > kSparseMaxKBlocks)
    return fail(JFA_ERR_INVALID_ARG, "block-sparse: max_len must be <= %d", kSparseMaxKBlocks * kBN);
  if (!blocks || !counts || (reinterpret_cast<uintptr_t>(blocks) & 3u) ||
      (reinterpret_cast<uintptr_t>(counts) & 3u))
    return fail(JFA_ERR_INVALID_ARG, "blocks and counts must be non-null, 4-byte aligned");
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != JFA_OK) return st;
  if (max_len == 0) {  // no Q block anywhere: nothing to write
    return finish(stream);
  }
  const size_t kbar_bytes = align256((size_t)B * H_kv * kcap * D * sizeof(float));
  const size_t bytes =
      kbar_bytes + align256((size_t)(s.broadcast ? 1 : B) * H * 2 * nqb * D * sizeof(float));
  void* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, bytes, ds->pool, stream);
  if (e != cudaSuccess) return fail(JFA_ERR_WORKSPACE, "scratch allocation: %s", cudaGetErrorString(e));
  SparseParams sp;
  memset(&sp, 0, sizeof(sp));
  sp.q = static_cast<const __nv_bfloat16*>(q);
  sp.k = static_cast<const __nv_bfloat16*>(k);
  sp.offsets = offsets;
  sp.B = B;
  sp.H = H;
  sp.Hkv = H_kv;
  sp.G = s.G;
  sp.D = D;
  sp.max_len = max_len;
  sp.permille = permille;
  sp.Lq = s.Lq;
  sp.broadcast = s.broadcast;
  sp.nqb = (int)nqb;
  sp.kcap = (int)kcap;
  sp.wl = s.kwl;
  sp.wr = s.kwr;
  sp.kbar = static_cast<float*>(scratch);
  sp.qsum = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + kbar_bytes);
  sp.blocks = blocks;
  sp.counts = counts;
  sp.err = ds->err;
  e = run_kernel(JFA_KERNEL_SPARSE_POOL, stream, [&] { return launch_sparse_pool(sp, stream); });
  if (e == cudaSuccess)
    e = run_kernel(JFA_KERNEL_SPARSE_SELECT, stream, [&] { return launch_sparse_select(sp, stream); });
  cudaError_t e2 = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "block selection launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch free");
  return finish(stream);
}

jfa_status jfa_fwd_sparse(const void* q, const void* k, const void* v, const int32_t* offsets,
                          int B, int H, int H_kv, int D, int max_len, int q_len, int broadcast_q,
                          float scale, const int32_t* blocks, const int32_t* counts, void* out,
                          float* lse, cudaStream_t stream) {
  return jfa_fwd_sparse_ex(q, k, v, offsets, B, H, H_kv, D, max_len, q_len, broadcast_q, 0, -1, -1,
                           scale, blocks, counts, out, lse, stream);
}

jfa_status jfa_fwd_sparse_ex(const void* q, const void* k, const void* v, const int32_t* offsets,
                             int B, int H, int H_kv, int D, int max_len, int q_len,
                             int broadcast_q, int causal, int window_left, int window_right,
                             float scale, const int32_t* blocks, const int32_t* counts, void* out,
                             float* lse, cudaStream_t stream) {
  t_last_error.clear();
  const Shape s = make_shape(B, H, H_kv, D, max_len, q_len, broadcast_q, causal, window_left,
                             window_right, scale);
  jfa_status st = check_common(s, q, k, v, offsets);
  if (st != JFA_OK) return st;
  if (!out || !aligned16(out)) return fail(JFA_ERR_INVALID_ARG, "out must be non-null, 16-byte aligned");
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(JFA_ERR_INVALID_ARG, "lse must be non-null, 4-byte aligned");
  if (!blocks || !counts || (reinterpret_cast<uintptr_t>(blocks) & 3u) ||
      (reinterpret_cast<uintptr_t>(counts) & 3u))
    return fail(JFA_ERR_INVALID_ARG, "blocks and counts must be non-null, 4-byte aligned");
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != JFA_OK) return st;
  if (s.max_len == 0) {  // no keys anywhere (broadcast: every row O = 0, LSE = -inf)
    if (s.broadcast) {
      cudaError_t e = run_kernel(JFA_KERNEL_FILL, stream, [&] {
        return launch_fill_empty(
            static_cast<__nv_bfloat16*>(out), lse, (long long)s.B * s.Lq * s.H, s.D, stream);
      });
      if (e != cudaSuccess) return cuda_fail(e, "fill launch");
    }
    return finish(stream);
  }
  const long long kcap = cdivll(s.max_len, kBN);
  const long long nqb = cdivll(s.broadcast ? s.Lq : s.max_len, kFwdRows);
  const long long cap = (long long)s.H * s.B * nqb;
  if (cap >= (1LL << 31) || (long long)s.B * s.H * nqb * kcap >= (1LL << 40))
    return fail(JFA_ERR_INVALID_ARG, "work list too large");
  SchedParams sp{offsets, s.B, s.H, s.Lq, s.max_len, s.local, s.broadcast, 0, kFwdRows, nullptr,
                 (int)cap, nullptr, ds->err, s.kwl, s.kwr};
  sp.blocks = blocks;
  sp.counts = counts;
  sp.nqb = (int)nqb;
  sp.kcap = (int)kcap;
  sp.n_check = list_check_blocks(sp);
  const size_t items_off = 256;
  const size_t check_off = align256(items_off + cap * sizeof(Item));
  const size_t bytes = align256(check_off + sp.n_check * sizeof(int));
  CUtensorMap tq, tk, tv;
  if ((st = map_rows(&tq, q, s.D, s.H, s.broadcast ? s.Lq : s.Tcap, "q")) != JFA_OK) return st;
  if ((st = map_rows(&tk, k, s.D, s.Hkv, s.Tcap, "k")) != JFA_OK) return st;
  if ((st = map_rows(&tv, v, s.D, s.Hkv, s.Tcap, "v")) != JFA_OK) return st;
  void* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, bytes, ds->pool, stream);
  if (e != cudaSuccess) return fail(JFA_ERR_WORKSPACE, "scratch allocation: %s", cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  WorkHeader* hdr = reinterpret_cast<WorkHeader*>(base);
  Item* items = reinterpret_cast<Item*>(base + items_off);
  sp.items = items;
  sp.hdr = hdr;
  sp.check = reinterpret_cast<int*>(base + check_off);
  // Every list is checked (many CTAs) before the scheduler reads the
  // results; a bad list leaves the work list empty, so nothing is written.
  e = run_kernel(JFA_KERNEL_SPARSE_CHECK, stream, [&] { return launch_list_check(sp, stream); });
  if (e == cudaSuccess)
    e = run_kernel(JFA_KERNEL_SCHED, stream, [&] { return launch_sched(sp, stream); });
  if (e == cudaSuccess) {
    FwdParams fp;
    memset(&fp, 0, sizeof(fp));
    set_variant(fp, s);
    fp.offsets = offsets;
    fp.B = s.B;
    fp.H = s.H;
    fp.Lq = s.Lq;
    fp.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
    fp.out = static_cast<__nv_bfloat16*>(out);
    fp.lse = lse;
    fp.items = items;
    fp.hdr = hdr;
    fp.err = ds->err;
    fp.blocks = blocks;
    fp.counts = counts;
    fp.nqb = (int)nqb;
    fp.kcap = (int)kcap;
    e = run_kernel(JFA_KERNEL_FWD, stream, [&] {
      return launch_fwd(s.D, s.local, s.broadcast, tq, tk, tv, fp, (int)cap, stream, true);
    });
  }
  cudaError_t e2 = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch free");
  return finish(stream);
}

jfa_status jfa_worklist(const int32_t* offsets, int B, int H, int max_len, int q_len,
                        int broadcast_q, int causal, int list, int32_t* items, int capacity,
                        int32_t* count, cudaStream_t stream) {
  t_last_error.clear();
  if (B < 1 || H < 1 || H > kMaxHeads || max_len < 0 || capacity < 0)
    return fail(JFA_ERR_INVALID_ARG, "worklist: B >= 1, 1 <= H <= %d, max_len, capacity >= 0",
                kMaxHeads);
  if (!offsets || (reinterpret_cast<uintptr_t>(offsets) & 3u) || !count ||
      (reinterpret_cast<uintptr_t>(count) & 3u) || (capacity > 0 && !aligned16(items)))
    return fail(JFA_ERR_INVALID_ARG, "worklist: offsets, count 4-byte and items 16-byte aligned");
  if (list < 0 || list > 3) return fail(JFA_ERR_INVALID_ARG, "worklist: list must be 0..3");
  if (broadcast_q && (causal || q_len < 1))
    return fail(JFA_ERR_INVALID_ARG, "worklist: broadcast needs q_len >= 1 and no causal mask");
  if ((list == 2 && broadcast_q) || (list == 3 && !broadcast_q))
    return fail(JFA_ERR_INVALID_ARG, "worklist: list 2 is self-attention only, 3 broadcast only");
  if ((long long)B * max_len >= (1LL << 31) || cdivll(max_len, kBN) > 65535)
    return fail(JFA_ERR_INVALID_ARG, "worklist: sequence lengths too large");
  DeviceState* ds = nullptr;
  jfa_status st = device_state(&ds);
  if (st != JFA_OK) return st;
  const int Lq = broadcast_q ? q_len : 0;
  long long cap = 0, chunk_cap = 0;
  const long long pairs = cdivll(Lq, kQbRows);
  if (list == 0)
    cap = (long long)H * B * (broadcast_q ? cdivll(Lq, kFwdRows) : cdivll(max_len, kFwdRows));
  else if (list == 1)
    cap = (long long)H * B * cdivll(max_len, kBN);
  else if (list == 2)
    cap = (long long)H * B * cdivll(max_len, kFwdRows);
  else {
    chunk_cap = std::max<long long>(1, cdivll(2LL * ds->sms, H * pairs));
    cap = chunk_cap * H * pairs;
  }
  if (cap >= (1LL << 31)) return fail(JFA_ERR_INVALID_ARG, "worklist: list too large");
  if (cap > capacity)
    return fail(JFA_ERR_INVALID_ARG, "worklist: items must hold %lld entries (4 ints each)", cap);
  const size_t item_bytes = list == 3 ? sizeof(QbItem) : sizeof(Item);
  const size_t ktoff = align256(256 + cap * item_bytes);
  const size_t bytes = align256(ktoff + (B + 1) * sizeof(int));
  void* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&scratch, bytes, ds->pool, stream);
  if (e != cudaSuccess) return fail(JFA_ERR_WORKSPACE, "scratch allocation: %s", cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(scratch);
  WorkHeader* hdr = reinterpret_cast<WorkHeader*>(base);
  void* list_items = base + 256;
  const int c = causal ? 1 : 0, bq = broadcast_q ? 1 : 0;
  if (list == 3) {
    QbSchedParams qp{offsets, B, H, Lq, max_len, (int)chunk_cap, reinterpret_cast<int*>(base + ktoff),
                     static_cast<QbItem*>(list_items), (int)cap, hdr, ds->err};
    e = run_kernel(JFA_KERNEL_PREP, stream, [&] { return launch_qb_sched(qp, stream); });
  } else {
    const int backward = list == 1 ? 1 : 0;
    SchedParams sp{offsets, B, H, Lq, max_len, c, bq, backward, backward ? kBM : kFwdRows,
                   static_cast<Item*>(list_items), (int)cap, hdr, ds->err};
    e = run_kernel(list == 0 ? JFA_KERNEL_SCHED : JFA_KERNEL_PREP, stream,
                   [&] { return launch_sched(sp, stream); });
  }
  if (e == cudaSuccess)
    e = launch_export_list(hdr, list_items, list == 3 ? 1 : 0, items, capacity, count, stream);
  cudaError_t e2 = cudaFreeAsync(scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "worklist launch");
  if (e2 != cudaSuccess) return cuda_fail(e2, "scratch free");
  return finish(stream);
}

long long jfa_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

jfa_status jfa_profile_enable(int on) {
  g_profile_on.store(on ? 1 : 0, std::memory_order_relaxed);
  return JFA_OK;
}

jfa_status jfa_profile_select(unsigned int kinds) {
  g_profile_kinds.store(kinds, std::memory_order_relaxed);
  return JFA_OK;
}

jfa_status jfa_profile_read(double* ms, long long* launches, int n) {
  if (n < 0 || (n > 0 && (ms == nullptr || launches == nullptr)))
    return fail(JFA_ERR_INVALID_ARG, "profile_read: n must be >= 0 and the arrays non-null");
  for (int i = 0; i < n; ++i) {
    ms[i] = 0.0;
    launches[i] = 0;
  }
  std::vector<ProfRecord> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  jfa_status st = JFA_OK;
  for (const ProfRecord& r : recs) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.start, r.stop);
    if (e != cudaSuccess) {
      if (st == JFA_OK) st = cuda_fail(e, "profile event");
    } else if (r.kind < n) {
      ms[r.kind] += t;
      launches[r.kind] += 1;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  return st;
}

jfa_status jfa_sync_and_check(cudaStream_t stream) {
  // Touches neither the scratch pool nor any other per-device state, so that
  // callers of the allocation-free entry point can use it too.
  return sync_and_read_error_word(stream);
}

const char* jfa_last_error(void) { return t_last_error.c_str(); }

const char* jfa_version(void) { return "jfa-gb300 0.2 (sm_103a)"; }

}  // extern "C"

namespace {

// Synchronise `stream`, then read and clear the current device's error
// word.  Allocates nothing (a synchronous copy into a host int).
jfa_status sync_and_read_error_word(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (word != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
    if (word & kErrTimeout)
      return fail(JFA_ERR_TIMEOUT, "a device-side bounded wait ran out (error bits 0x%x)", word);
    if (word & kErrBadBlocks)
      return fail(JFA_ERR_INVALID_ARG,
                  "a block-sparse list failed device checks: a count above the sequence's key "
                  "tiles, or entries not strictly ascending below it (error bits 0x%x)",
                  word);
    if (word & kErrBadOffsets)
      return fail(JFA_ERR_INVALID_ARG,
                  "offsets failed device checks: offsets[0] != 0, decreasing, or a length above "
                  "max_len (error bits 0x%x)",
                  word);
    return fail(JFA_ERR_CUDA, "device error bits 0x%x", word);
  }
  return JFA_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Allocation-free forward entry point.
//
// Some callers may not allocate device memory at all while they run this
// library: code whose memory is entirely owned and pre-partitioned by a host
// framework (inference servers and plugin hosts that hand a library fixed
// buffers and forbid allocations during execution), real-time loops that
// must not take the allocator's locks or risk an out-of-memory failure
// mid-run, and code running where the caller has made allocation illegal.
// For them the forward pass keeps its scratch (the work-list header and the
// work items) in the file-scope device array below instead of a pool.
// ---------------------------------------------------------------------------

namespace {

// Maximum scratch of the allocation-free forward: 256 B header plus 8 B per
// work item, i.e. at most (1 MiB - 256 B) / 8 = 131040 items, where items =
// H * B * ceil(max_len / 256) (self-attention) or H * B * ceil(q_len / 256)
// (broadcast-Q).  Every GPU that loads the library holds this array until
// the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  int sms = 0;
  int* err = nullptr;          // device address of the error word
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch
};
NoAllocDevice g_noalloc_dev[kMaxDevices];

// Once per device, with that device current: resolve the device addresses of
// the scratch array and of the error word.  In host code the array's name is
// only a host-side stand-in, so its address must come from
// cudaGetSymbolAddress.  Nothing here allocates memory.
jfa_status noalloc_device(NoAllocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(JFA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(JFA_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess)
      return fail(JFA_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
    if (!(prop.major == 10 && prop.minor == 3))
      return fail(JFA_ERR_UNSUPPORTED, "device %s is sm_%d%d; this library is built for sm_103a",
                  prop.name, prop.major, prop.minor);
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(JFA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    void* err = nullptr;
    e = cudaGetSymbolAddress(&err, g_device_error);
    if (e != cudaSuccess || err == nullptr)
      return fail(JFA_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || !fn || q != cudaDriverEntryPointSuccess)
        return fail(JFA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.sms = prop.multiProcessorCount;
    d.scratch = static_cast<uint8_t*>(ptr);
    d.err = static_cast<int*>(err);
    d.ready = true;
  }
  *out = &d;
  return JFA_OK;
}

}  // namespace

extern "C" {

jfa_status jfa_fwd_bq_noalloc(const void* q, const void* k, const void* v, const int32_t* offsets,
                              int B, int H, int D, int max_len, int q_len, int broadcast_q,
                              int causal, float scale, void* out, float* lse,
                              cudaStream_t stream) {
  t_last_error.clear();
  const Shape s = make_shape(B, H, H, D, max_len, q_len, broadcast_q, causal, -1, -1, scale);
  jfa_status st = check_common(s, q, k, v, offsets);
  if (st != JFA_OK) return st;
  if (!out || !aligned16(out)) return fail(JFA_ERR_INVALID_ARG, "out must be non-null, 16-byte aligned");
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(JFA_ERR_INVALID_ARG, "lse must be non-null, 4-byte aligned");
  const long long qt = s.broadcast ? cdivll(s.Lq, kFwdRows) : cdivll(s.max_len, kFwdRows);
  const long long cap = (long long)s.H * s.B * qt;
  const size_t items_off = 256;
  const long long max_items = (long long)((kNoAllocScratchBytes - items_off) / sizeof(Item));
  if (cap > max_items)
    return fail(JFA_ERR_WORKSPACE,
                "jfa_fwd_bq_noalloc: this problem needs up to %lld work items (H * B * "
                "ceil(len / 256)) but the static scratch array (%zu bytes) holds at most %lld; "
                "use jfa_fwd / jfa_fwd_bq",
                cap, kNoAllocScratchBytes, max_items);
  NoAllocDevice* d = nullptr;
  if ((st = noalloc_device(&d)) != JFA_OK) return st;
  cudaError_t e;
  if (s.max_len == 0) {
    if (s.broadcast) {
      e = run_kernel(JFA_KERNEL_FILL, stream, [&] {
        return launch_fill_empty(
            static_cast<__nv_bfloat16*>(out), lse, (long long)s.B * s.Lq * s.H, s.D, stream);
      });
      if (e != cudaSuccess) return cuda_fail(e, "fill launch");
    }
    return finish(stream);
  }
  CUtensorMap tq, tk, tv;
  if ((st = map_rows(&tq, q, s.D, s.H, s.broadcast ? s.Lq : s.Tcap, "q")) != JFA_OK) return st;
  if ((st = map_rows(&tk, k, s.D, s.H, s.Tcap, "k")) != JFA_OK) return st;
  if ((st = map_rows(&tv, v, s.D, s.H, s.Tcap, "v")) != JFA_OK) return st;
  WorkHeader* hdr = reinterpret_cast<WorkHeader*>(d->scratch);
  Item* items = reinterpret_cast<Item*>(d->scratch + items_off);
  // The scheduler rewrites the header (item count, T, ticket = 0) and every
  // item the forward kernel reads, so nothing left by a previous call leaks.
  SchedParams sp{offsets, s.B, s.H, s.Lq, s.max_len, s.causal, s.broadcast, 0, kFwdRows,
                 items, (int)cap, hdr, d->err};
  e = run_kernel(JFA_KERNEL_SCHED, stream, [&] {
    return launch_sched(sp, stream);
  });
  if (e != cudaSuccess) return cuda_fail(e, "scheduler launch");
  FwdParams fp;
  memset(&fp, 0, sizeof(fp));
  set_variant(fp, s);
  fp.offsets = offsets;
  fp.B = s.B;
  fp.H = s.H;
  fp.Lq = s.Lq;
  fp.scale_log2 = (float)((double)s.scale * 1.4426950408889634);
  fp.out = static_cast<__nv_bfloat16*>(out);
  fp.lse = lse;
  fp.items = items;
  fp.hdr = hdr;
  fp.err = d->err;
  const int grid = (int)cap;  // one CTA per possible item (cluster launch control)
  e = run_kernel(JFA_KERNEL_FWD, stream, [&] {
    return launch_fwd(s.D, s.causal, s.broadcast, tq, tk, tv, fp, grid, stream);
  });
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return finish(stream);
}


}  // extern "C"
