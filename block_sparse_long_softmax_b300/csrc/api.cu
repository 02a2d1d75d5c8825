// C ABI of libskipsm: argument validation, tensor maps, launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/skipsm.h"
#include "internal.h"

namespace skipsm {

__device__ int g_device_status = 0;

#if SKIPSM_TRACE
// Test-only instrumentation: the next prefill launches stamp the events of CTA
// `g_trace_cta` into `g_trace_buf` (see skipsm_debug_prefill_trace).
unsigned long long* g_trace_buf = nullptr;
int g_trace_cta = -1;
unsigned long long* g_decode_trace_buf = nullptr;
#endif

namespace {

thread_local char t_last_error[512] = "";

skipsm_status fail(skipsm_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return st;
}

skipsm_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SKIPSM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- driver entry point for tensor-map encoding (no libcuda link needed)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor [Z][S][D] (D innermost) seen as 3-D with a (64 x rows x 1) box
// and 128-byte swizzle; out-of-range elements read as zero.
// 3-D map (D, S, Z) of a [Z][S][D] tensor of bf16 (elem = 2) or 8-bit (elem = 1) values;
// the box is one 128-byte swizzle row of D by box_rows rows.
skipsm_status make_map(CUtensorMap* m, const void* base, int D, long long S, long long Z,
                       int box_rows, int elem = 2) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(SKIPSM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(Z)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elem, static_cast<cuuint64_t>(S) * D * elem};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                   3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SKIPSM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return SKIPSM_OK;
}

long long wait_cycles(int ms) {
  if (ms <= 0) ms = 2000;
  return static_cast<long long>(ms) * 2100000LL;  // upper SM clock, 2.1 GHz
}

skipsm_status check_lambda(float lambda) {
  if (!std::isfinite(lambda) || lambda < 0.f || lambda > 1.f)
    return fail(SKIPSM_ERR_INVALID_ARG, "lambda must be finite and in [0, 1] (got %g)", lambda);
  return SKIPSM_OK;
}

void set_lambda(float lambda, float* lam_log2, int* lam_pos) {
  *lam_pos = lambda > 0.f;
  *lam_log2 = lambda > 0.f ? static_cast<float>(std::log2(static_cast<double>(lambda))) : -INFINITY;
}

constexpr int kDecodeBk = 64;
// Default split count: split CTAs run in waves of (SMs) * kDecodeCtasPerSm (two
// resident per SM at D = 128, bound by shared memory), and a wave that is only partly
// filled costs nearly as much as a full one.  Each CTA also pays a start-up of about
// kDecodeCtaStartTiles tile loads before its pipeline is full.  The SM count is read
// from the device; kDecodeSms (B300) stands in when no device can be queried.
constexpr int kDecodeSms = 148;
constexpr int kDecodeCtasPerSm = 2;
constexpr int kDecodeCtaStartTiles = 4;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int device_sm_count() {
  static std::atomic<int> counts[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();  // no device here: clear the error, use the B300 count
    return kDecodeSms;
  }
  int n = counts[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return kDecodeSms;
    }
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int* device_status_word() {
  // One slot per device, keyed by the context it was looked up in: a device reset or
  // another context on the device gets its own lookup.
  struct Slot { unsigned long long ctx; int* ptr; };
  static std::mutex mu;
  static Slot slots[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long ctx = current_context_id();
  if (!slots[dev].ptr || ctx == 0 || slots[dev].ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    // the lookup made the device's primary context current if none was
    if (ctx == 0) ctx = current_context_id();
    slots[dev] = Slot{ctx, static_cast<int*>(p)};
  }
  return slots[dev].ptr;
}

}  // namespace skipsm

using namespace skipsm;

extern "C" {

int skipsm_version(void) { return SKIPSM_VERSION; }

#if SKIPSM_TRACE
// Only in SKIPSM_TRACE builds (libskipsm_trace.so): later prefill calls record clock64
// stamps of CTA `cta` into `buf` (device, [key tiles][2][16] uint64, zeroed by the
// caller); buf = NULL stops recording.  Not part of the library's interface.
void skipsm_debug_prefill_trace(void* buf, int cta) {
  g_trace_buf = static_cast<unsigned long long*>(buf);
  g_trace_cta = cta;
}
// Only in SKIPSM_TRACE builds: later decode calls record the start and end times
// (%globaltimer, ns) of every split CTA into `buf` (device, [B][Hkv][splits][2] uint64);
// buf = NULL stops recording.  Not part of the library's interface.
void skipsm_debug_decode_trace(void* buf) {
  g_decode_trace_buf = static_cast<unsigned long long*>(buf);
}
#endif

const char* skipsm_last_error(void) { return t_last_error; }

skipsm_status skipsm_check(void* stream, int* device_status) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int* w = device_status_word();
  if (!w) return fail(SKIPSM_ERR_CUDA, "device status word unavailable");
  int v = 0;
  e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device status");
  if (v) {
    const int zero = 0;
    e = cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device status");
  }
  if (device_status) *device_status = v;
  if (v) return fail(SKIPSM_ERR_TIMEOUT, "a kernel wait exceeded its bound (site %d)", v);
  t_last_error[0] = '\0';
  return SKIPSM_OK;
}

// The sync_check option: wait for the stream, then report the call's device status (its own
// word, left as it is, or the shared word, read and cleared as by skipsm_check).
static skipsm_status sync_and_check(cudaStream_t s, int* own) {
  if (!own) return skipsm_check(s, nullptr);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, own, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status");
  if (v) return fail(SKIPSM_ERR_TIMEOUT, "a kernel wait exceeded its bound (site %d)", v);
  t_last_error[0] = '\0';
  return SKIPSM_OK;
}

// ------------------------------------------------------------------ prefill
skipsm_status skipsm_prefill_ex(const void* q, const void* k, const void* v, void* o, int B,
                                int Hq, int Hkv, int Sq, int Skv, int D, int causal, float lambda,
                                uint64_t* skip_counts, const skipsm_prefill_opts* opts,
                                void* stream) {
  skipsm_prefill_opts op;
  std::memset(&op, 0, sizeof(op));
  if (opts) op = *opts;
  if (!q || !k || !v || !o) return fail(SKIPSM_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(SKIPSM_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1)
    return fail(SKIPSM_ERR_INVALID_ARG, "sizes must be >= 1");
  if (Hq % Hkv) return fail(SKIPSM_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (D != 64 && D != 128) return fail(SKIPSM_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", D);
  if (causal && Sq > Skv) return fail(SKIPSM_ERR_INVALID_ARG, "causal prefill needs Sq <= Skv");
  skipsm_status st = check_lambda(lambda);
  if (st) return st;
  const int tq = op.tile_q ? op.tile_q : (D == 64 ? 64 : 128);
  const int tk = op.tile_k ? op.tile_k : (D == 64 ? 64 : 128);
  if ((tq != 64 && tq != 128) || (tk != 64 && tk != 128))
    return fail(SKIPSM_ERR_UNSUPPORTED, "tile_q / tile_k must be 64 or 128");
  if (!(op.softmax_scale >= 0.f) || !std::isfinite(op.softmax_scale))
    return fail(SKIPSM_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  if (op.exp_mode != 0 && op.exp_mode != 1)
    return fail(SKIPSM_ERR_INVALID_ARG, "exp_mode must be 0 (exact) or 1 (Rowmax-PoT)");
  if (op.qk_format != 0 && op.qk_format != 1)
    return fail(SKIPSM_ERR_INVALID_ARG, "qk_format must be 0 (bf16) or 1 (e4m3)");
  if (op.qk_format == 1 && (D != 128 || tk != 128))
    return fail(SKIPSM_ERR_UNSUPPORTED, "e4m3 q/k need D = 128 and tile_k = 128");
  if (!(op.qk_descale >= 0.f) || !std::isfinite(op.qk_descale))
    return fail(SKIPSM_ERR_INVALID_ARG, "qk_descale must be finite and >= 0");
  if (op.v_format != 0 && op.v_format != 1)
    return fail(SKIPSM_ERR_INVALID_ARG, "v_format must be 0 (bf16) or 1 (e4m3, transposed)");
  if (op.v_format == 1 && (op.qk_format != 1 || op.exp_mode != 0))
    return fail(SKIPSM_ERR_UNSUPPORTED, "e4m3 v needs e4m3 q/k and exact exponentials");
  if (op.v_format == 1 && Skv % 16)
    return fail(SKIPSM_ERR_UNSUPPORTED, "e4m3 v needs Skv to be a multiple of 16 (row stride)");
  if (!(op.v_descale >= 0.f) || !std::isfinite(op.v_descale))
    return fail(SKIPSM_ERR_INVALID_ARG, "v_descale must be finite and >= 0");
  if (op.v_load < 0 || op.v_load > 2)
    return fail(SKIPSM_ERR_INVALID_ARG, "v_load must be 0, 1 or 2");
  const long long nblk_q = (Sq + 255) / 256;
  if (nblk_q * B * Hq > 0x7FFFFFFFLL) return fail(SKIPSM_ERR_UNSUPPORTED, "grid too large");
  int* status = op.status ? op.status : device_status_word();
  if (!status) return fail(SKIPSM_ERR_CUDA, "device status word unavailable");
  if (reinterpret_cast<uintptr_t>(status) & 3u)
    return fail(SKIPSM_ERR_INVALID_ARG, "status must be 4-byte aligned");

  CUtensorMap qmap, kmap, vmap;
  const int qk_elem = op.qk_format == 1 ? 1 : 2;
  if ((st = make_map(&qmap, q, D, Sq, static_cast<long long>(B) * Hq, 128, qk_elem))) return st;
  if ((st = make_map(&kmap, k, D, Skv, static_cast<long long>(B) * Hkv, tk, qk_elem))) return st;
  if (op.v_format == 1) {
    // v^T [B*Hkv][D][Skv]: boxes of 128 keys (one 128-byte atom) by D rows
    if ((st = make_map(&vmap, v, Skv, D, static_cast<long long>(B) * Hkv, D, 1))) return st;
  } else if ((st = make_map(&vmap, v, D, Skv, static_cast<long long>(B) * Hkv, tk))) {
    return st;
  }

  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.Sq = Sq; p.Skv = Skv; p.D = D;
  p.causal = causal ? 1 : 0;
  p.tile_q = tq; p.tile_k = tk;
  p.nqt = (Sq + tq - 1) / tq;
  p.nkt = (Skv + tk - 1) / tk;
  p.nblk_q = static_cast<int>(nblk_q);
  const double scale = (op.softmax_scale > 0.f ? op.softmax_scale : 1.0 / std::sqrt((double)D)) *
                       (op.qk_descale > 0.f ? op.qk_descale : 1.0);
  p.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  set_lambda(lambda, &p.lam_log2, &p.lam_pos);
  p.qk_e4m3 = op.qk_format == 1 ? 1 : 0;
  p.v_e4m3 = op.v_format == 1 ? 1 : 0;
  p.v_descale = op.v_descale > 0.f ? op.v_descale : 1.f;
  p.v_after_vote = op.v_load == 2 ? 1 : 0;
  p.block_mask = op.block_mask;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = op.lse;
  p.skip_counts = reinterpret_cast<unsigned long long*>(skip_counts);
  p.visited_counts = reinterpret_cast<unsigned long long*>(op.visited_counts);
  p.skip_mask = op.skip_mask;
  p.status = status;
  p.wait_cycles = wait_cycles(op.wait_limit_ms);
  p.exp_mode = op.exp_mode;
  p.inject_fault = op.inject_wait_timeout ? 1 : 0;
#if SKIPSM_TRACE
  p.trace = g_trace_buf;
  p.trace_cta = g_trace_cta;
#endif

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (skip_counts && (e = cudaMemsetAsync(skip_counts, 0, sizeof(uint64_t) * Hq, s)))
    return cuda_fail(e, "zero skip_counts");
  if (op.visited_counts && (e = cudaMemsetAsync(op.visited_counts, 0, sizeof(uint64_t) * Hq, s)))
    return cuda_fail(e, "zero visited_counts");
  if (op.skip_mask &&
      (e = cudaMemsetAsync(op.skip_mask, 2, static_cast<size_t>(B) * Hq * p.nqt * p.nkt, s)))
    return cuda_fail(e, "init skip_mask");
  if ((e = launch_prefill(qmap, kmap, vmap, p, s))) return cuda_fail(e, "prefill launch");
  if (op.sync_check) return sync_and_check(s, op.status);
  return SKIPSM_OK;
}

skipsm_status skipsm_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                             int Hkv, int Sq, int Skv, int D, int causal, float lambda,
                             uint64_t* skip_counts, void* stream) {
  return skipsm_prefill_ex(q, k, v, o, B, Hq, Hkv, Sq, Skv, D, causal, lambda, skip_counts,
                           nullptr, stream);
}

// ------------------------------------------------------------------- decode
int skipsm_decode_num_splits(int B, int Hkv, int Skv, int requested) {
  if (B < 1 || Hkv < 1 || Skv < 1 || requested < 0) return 0;
  const int nblk = (Skv + kDecodeBk - 1) / kDecodeBk;
  int want = requested;
  if (want == 0) {
    // The count with the least modelled time: waves x (tiles per split + start-up), the
    // fewest splits on a tie.  Fewer splits also skip more: each split's first tile is
    // always kept (its running max starts at -inf), and a split that has not yet seen
    // the large logits of earlier keys keeps tiles a longer prefix would skip.  Splits
    // hold at least 16 tiles.
    const long long items = static_cast<long long>(B) * Hkv;
    const long long slots = static_cast<long long>(device_sm_count()) * kDecodeCtasPerSm;
    const int hi = static_cast<int>(std::min<long long>(std::max(1, nblk / 16), slots * 8));
    long long best = -1;
    want = 1;
    for (int s = 1; s <= hi; ++s) {
      const int per = (nblk + s - 1) / s;
      if ((nblk + per - 1) / per != s) continue;  // the same cut as a smaller count
      const long long waves = (items * s + slots - 1) / slots;
      const long long cost = waves * (per + kDecodeCtaStartTiles);
      if (best < 0 || cost < best) {
        best = cost;
        want = s;
      }
    }
  }
  want = std::max(1, std::min(want, nblk));
  const int per = (nblk + want - 1) / want;
  return (nblk + per - 1) / per;
}

size_t skipsm_decode_workspace_size(int B, int Hq, int Hkv, int Skv, int D, int num_splits) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1) return 0;
  const int ns = skipsm_decode_num_splits(B, Hkv, Skv, num_splits);
  if (ns == 0) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * ns;
  return align256(rows * D * sizeof(float)) + align256(rows * sizeof(float));
}

skipsm_status skipsm_decode_ex(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                               int Hkv, int Skv, int D, float lambda, uint64_t* skip_counts,
                               void* workspace, size_t workspace_bytes,
                               const skipsm_decode_opts* opts, void* stream) {
  skipsm_decode_opts op;
  std::memset(&op, 0, sizeof(op));
  if (opts) op = *opts;
  if (!q || !k || !v || !o) return fail(SKIPSM_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(SKIPSM_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (B < 1 || Hq < 1 || Hkv < 1 || Skv < 1) return fail(SKIPSM_ERR_INVALID_ARG, "sizes must be >= 1");
  if (Hq % Hkv) return fail(SKIPSM_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(SKIPSM_ERR_UNSUPPORTED, "decode GQA group %d (supported: 1, 2, 4, 8)", G);
  if (D != 64 && D != 128) return fail(SKIPSM_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", D);
  skipsm_status st = check_lambda(lambda);
  if (st) return st;
  if (op.num_splits < 0) return fail(SKIPSM_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (!(op.softmax_scale >= 0.f) || !std::isfinite(op.softmax_scale))
    return fail(SKIPSM_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  if (static_cast<long long>(B) * Hkv > 65535LL * 65535LL)
    return fail(SKIPSM_ERR_UNSUPPORTED, "grid too large");
  if (B > 65535 || Hkv > 65535) return fail(SKIPSM_ERR_UNSUPPORTED, "B and Hkv must be <= 65535");
  const int ns = skipsm_decode_num_splits(B, Hkv, Skv, op.num_splits);
  const size_t need = skipsm_decode_workspace_size(B, Hq, Hkv, Skv, D, op.num_splits);
  if (!workspace || workspace_bytes < need)
    return fail(SKIPSM_ERR_WORKSPACE, "decode needs %zu bytes of workspace (got %zu)", need,
                workspace_bytes);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(SKIPSM_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  int* status = op.status ? op.status : device_status_word();
  if (!status) return fail(SKIPSM_ERR_CUDA, "device status word unavailable");
  if (reinterpret_cast<uintptr_t>(status) & 3u)
    return fail(SKIPSM_ERR_INVALID_ARG, "status must be 4-byte aligned");

  CUtensorMap kmap, vmap;
  if ((st = make_map(&kmap, k, D, Skv, static_cast<long long>(B) * Hkv, kDecodeBk))) return st;
  if ((st = make_map(&vmap, v, D, Skv, static_cast<long long>(B) * Hkv, kDecodeBk))) return st;

  const int nblk = (Skv + kDecodeBk - 1) / kDecodeBk;
  const size_t rows = static_cast<size_t>(B) * Hq * ns;
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.Skv = Skv; p.D = D;
  p.nblk = nblk;
  p.per = (nblk + ns - 1) / ns;
  p.nsplit = ns;
  const double scale = op.softmax_scale > 0.f ? op.softmax_scale : 1.0 / std::sqrt((double)D);
  p.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  set_lambda(lambda, &p.lam_log2, &p.lam_pos);
  p.ws_o = static_cast<float*>(workspace);
  p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * D * sizeof(float)));
  p.skip_counts = reinterpret_cast<unsigned long long*>(skip_counts);
  p.skip_mask = op.skip_mask;
  p.status = status;
  p.wait_cycles = wait_cycles(op.wait_limit_ms);
  p.inject_fault = op.inject_wait_timeout ? 1 : 0;
  p.block_mask = op.block_mask;
#if SKIPSM_TRACE
  p.trace = g_decode_trace_buf;
#endif
  cudaError_t e;
  if (p.block_mask) {
    int dev = 0, optin = 0;
    if ((e = cudaGetDevice(&dev)) ||
        (e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
      return cuda_fail(e, "query shared memory limit");
    if (decode_smem_bytes(p) > static_cast<size_t>(optin))
      return fail(SKIPSM_ERR_UNSUPPORTED,
                  "block mask: a split of %d tiles does not fit in shared memory; use more splits",
                  p.per);
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (skip_counts && (e = cudaMemsetAsync(skip_counts, 0, sizeof(uint64_t) * Hq, s)))
    return cuda_fail(e, "zero skip_counts");
  if (p.block_mask && op.skip_mask &&
      (e = cudaMemsetAsync(op.skip_mask, 2, static_cast<size_t>(B) * Hkv * nblk, s)))
    return cuda_fail(e, "initialise skip_mask");
  if ((e = launch_decode(kmap, vmap, p, B, s))) return cuda_fail(e, "decode split launch");
  CombineParams c;
  c.ws_o = p.ws_o;
  c.ws_lse = p.ws_lse;
  c.o = static_cast<__nv_bfloat16*>(o);
  c.lse = op.lse;
  c.Hq = Hq; c.D = D; c.nsplit = ns;
  if ((e = launch_combine(c, B, s))) return cuda_fail(e, "decode combine launch");
  if (op.sync_check) return sync_and_check(s, op.status);
  return SKIPSM_OK;
}

skipsm_status skipsm_decode(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                            int Hkv, int Skv, int D, float lambda, uint64_t* skip_counts,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return skipsm_decode_ex(q, k, v, o, B, Hq, Hkv, Skv, D, lambda, skip_counts, workspace,
                          workspace_bytes, nullptr, stream);
}

// -------------------------------------------------------------- calibration
}  // extern "C"

namespace {

// Bisection on log10(lambda) in [-9, 0] for the lambda whose skip ratio is closest
// to `target`; `run(lambda, &ratio)` performs one attention call and measures it.
template <class Run>
skipsm_status bisect_lambda(float target, int max_iters, Run run, skipsm_calibration* res) {
  if (!res) return fail(SKIPSM_ERR_INVALID_ARG, "result pointer is NULL");
  if (!(target >= 0.f && target <= 1.f))
    return fail(SKIPSM_ERR_INVALID_ARG, "target skip ratio must be in [0, 1]");
  if (max_iters < 0 || max_iters > 64) return fail(SKIPSM_ERR_INVALID_ARG, "max_iters in [0, 64]");
  if (max_iters == 0) max_iters = 14;
  double lo = -9.0, hi = 0.0;
  float best_l = 0.f, best_r = 0.f;
  double best_d = 2.0;
  int launches = 0;
  for (int it = 0; it < max_iters; ++it) {
    const double mid = 0.5 * (lo + hi);
    const float lam = static_cast<float>(std::pow(10.0, mid));
    float ratio = 0.f;
    const skipsm_status st = run(lam, &ratio);
    ++launches;
    if (st != SKIPSM_OK) return st;
    const double d = std::fabs(static_cast<double>(ratio) - target);
    if (d < best_d) { best_d = d; best_l = lam; best_r = ratio; }
    if (ratio < target) lo = mid; else hi = mid;
  }
  res->lambda = best_l;
  res->skip_ratio = best_r;
  res->launches = launches;
  return SKIPSM_OK;
}

skipsm_status read_counts(const uint64_t* dev, int n, std::vector<uint64_t>* host, cudaStream_t s) {
  host->resize(n);
  cudaError_t e = cudaMemcpyAsync(host->data(), dev, sizeof(uint64_t) * n, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "read skip counts");
  return SKIPSM_OK;
}

}  // namespace

extern "C" {

skipsm_status skipsm_prefill_calibrate(const void* q, const void* k, const void* v, void* o, int B,
                                       int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                                       float target_skip_ratio, int max_iters, uint64_t* counts,
                                       const skipsm_prefill_opts* opts,
                                       skipsm_calibration* result, void* stream) {
  if (!counts) return fail(SKIPSM_ERR_INVALID_ARG, "counts scratch is NULL");
  skipsm_prefill_opts op;
  std::memset(&op, 0, sizeof(op));
  if (opts) op = *opts;
  if (op.skip_mask || op.visited_counts || op.lse)
    return fail(SKIPSM_ERR_INVALID_ARG, "calibration takes no optional outputs");
  op.visited_counts = counts + Hq;
  std::vector<uint64_t> h;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto run = [&](float lam, float* ratio) -> skipsm_status {
    skipsm_status st = skipsm_prefill_ex(q, k, v, o, B, Hq, Hkv, Sq, Skv, D, causal, lam, counts,
                                         &op, stream);
    if (st != SKIPSM_OK) return st;
    if ((st = read_counts(counts, 2 * Hq, &h, s)) != SKIPSM_OK) return st;
    uint64_t sk = 0, vis = 0;
    for (int i = 0; i < Hq; ++i) { sk += h[i]; vis += h[Hq + i]; }
    *ratio = vis ? static_cast<float>(static_cast<double>(sk) / static_cast<double>(vis)) : 0.f;
    return SKIPSM_OK;
  };
  return bisect_lambda(target_skip_ratio, max_iters, run, result);
}

skipsm_status skipsm_decode_calibrate(const void* q, const void* k, const void* v, void* o, int B,
                                      int Hq, int Hkv, int Skv, int D, float target_skip_ratio,
                                      int max_iters, uint64_t* counts, void* workspace,
                                      size_t workspace_bytes, const skipsm_decode_opts* opts,
                                      skipsm_calibration* result, void* stream) {
  if (!counts) return fail(SKIPSM_ERR_INVALID_ARG, "counts scratch is NULL");
  skipsm_decode_opts op;
  std::memset(&op, 0, sizeof(op));
  if (opts) op = *opts;
  if (op.skip_mask || op.lse) return fail(SKIPSM_ERR_INVALID_ARG, "calibration takes no optional outputs");
  if (Hkv < 1 || Hq < Hkv || Hq % Hkv) return fail(SKIPSM_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  const int G = Hq / Hkv;
  const double tiles = static_cast<double>(B) * Hkv * ((Skv + kDecodeBk - 1) / kDecodeBk);
  std::vector<uint64_t> h;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto run = [&](float lam, float* ratio) -> skipsm_status {
    skipsm_status st = skipsm_decode_ex(q, k, v, o, B, Hq, Hkv, Skv, D, lam, counts, workspace,
                                        workspace_bytes, &op, stream);
    if (st != SKIPSM_OK) return st;
    if ((st = read_counts(counts, Hq, &h, s)) != SKIPSM_OK) return st;
    uint64_t sk = 0;
    for (int i = 0; i < Hq; i += G) sk += h[i];  // a group's count is repeated for its heads
    *ratio = tiles > 0 ? static_cast<float>(static_cast<double>(sk) / tiles) : 0.f;
    return SKIPSM_OK;
  };
  return bisect_lambda(target_skip_ratio, max_iters, run, result);
}

}  // extern "C"
