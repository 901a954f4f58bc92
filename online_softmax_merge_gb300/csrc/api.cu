// C ABI of libringattn.so (declared in include/ringattn.h): argument checks,
// status word, TMA tensor maps, and launches. No device memory is allocated
// here; the only device state is one static status word per GPU.
#include <math.h>
#include <string.h>

#include <atomic>
#include <initializer_list>
#include <mutex>
#include <new>

#include "internal.cuh"
#include "shardmap.cuh"

using namespace ra;

namespace ra {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<CtxGetCurrentFn>(a);
      get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace ra

namespace {
// The CUDA error behind the calling thread's most recent RA_ERR_CUDA (0 before any).
thread_local int32_t g_last_cuda_error = 0;
}  // namespace

ra_status ra::cuda_failed(cudaError_t e) {
  g_last_cuda_error = static_cast<int32_t>(e);
  return RA_ERR_CUDA;
}

namespace {

// Status word of the GPU: a kernel that gives up on a wait records its code here.
__device__ int g_status = 0;

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s for any single device-side wait
// The limit later launches get: kWaitLimitNs unless a test lowered it
// (ring_attn_selftest_wait_limit).
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
constexpr int kMaxDevices = 64;

struct DevInfo {
  bool init = false;
  bool sm103 = false;
  int ordinal = -1;
  unsigned long long ctx = 0;   // context the facts below were read in (0: unknown)
  int* status = nullptr;
};
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

// Current device's facts; RA_ERR_UNSUPPORTED unless it is compute capability 10.3.
// They are read again whenever the current context is not the one they were read in
// (the status word's device address belongs to a context).
ra_status current_device(DevInfo** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_failed(e);
  if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init || id == 0 || d.ctx != id) {
    d.init = false;
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_failed(e);
    d.sm103 = (major == 10 && minor == 3);
    d.ordinal = dev;
    d.status = nullptr;
    if (d.sm103) {
      void* ptr = nullptr;
      if ((e = cudaGetSymbolAddress(&ptr, g_status)) != cudaSuccess) {
        (void)cudaGetLastError();
        return cuda_failed(e);
      }
      d.status = static_cast<int*>(ptr);
    }
    d.ctx = current_context_id();   // the lookup made the device's context current
    d.init = true;
  }
  *out = &d;
  return d.sm103 ? RA_OK : RA_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The bytes [p, p + bytes) an argument covers.
struct Span {
  const void* p;
  size_t bytes;
};

bool overlap(const Span& a, const Span& b) {
  if (a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a.p), y = reinterpret_cast<uintptr_t>(b.p);
  return x < y + b.bytes && y < x + a.bytes;
}

// True when no range a call writes shares a byte with another written range or with a
// range it reads. Read ranges may overlap each other (the same tensor passed twice);
// a kernel writing where other CTAs still read would give undefined results.
bool writes_disjoint(std::initializer_list<Span> writes, std::initializer_list<Span> reads) {
  for (const Span* w = writes.begin(); w != writes.end(); ++w) {
    for (const Span& r : reads)
      if (overlap(*w, r)) return false;
    for (const Span* w2 = w + 1; w2 != writes.end(); ++w2)
      if (overlap(*w, *w2)) return false;
  }
  return true;
}

// Bytes of the tensors of a problem: q and o, k and v, one [B, H, N] fp32 row set
// (lse, m, z), and y.
struct Bytes {
  size_t q, kv, rows, y, o;
};
Bytes tensor_bytes(const ra_problem* pr) {
  const size_t tok = static_cast<size_t>(pr->batch) * static_cast<size_t>(pr->seqlen);
  Bytes b;
  b.q = tok * pr->heads * pr->head_dim * 2;
  b.kv = tok * pr->kv_heads * pr->head_dim * 2;
  b.rows = tok * pr->heads * sizeof(float);
  b.y = tok * pr->heads * pr->head_dim * sizeof(float);
  b.o = pr->o_dtype == RA_DTYPE_F32 ? b.y : b.q;
  return b;
}

// Memory the kernels launched on the current device may touch: device memory of that
// device (cudaMalloc, stream-ordered pools, virtual-memory mappings) or managed memory.
// Host memory (pageable or pinned) and other devices' memory are refused before
// anything is launched, since a kernel reading them could fault the GPU.
ra_status resident(const DevInfo* d, std::initializer_list<const void*> ptrs) {
  for (const void* ptr : ptrs) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
      (void)cudaGetLastError();   // the failed query leaves a (non-sticky) error behind
      return RA_ERR_INVALID_ARG;
    }
    const bool ok = a.type == cudaMemoryTypeManaged ||
                    (a.type == cudaMemoryTypeDevice && a.device == d->ordinal);
    if (!ok) return RA_ERR_INVALID_ARG;
  }
  return RA_OK;
}

ra_status check_layout_sizes(int32_t layout, int32_t seqlen, int32_t P) {
  if (layout != RA_LAYOUT_CONTIGUOUS && layout != RA_LAYOUT_STRIPED && layout != RA_LAYOUT_ZIGZAG)
    return RA_ERR_INVALID_ARG;
  if (seqlen < 1 || P < 1 || P > seqlen || seqlen % P != 0 || seqlen >= (1 << 30))
    return RA_ERR_INVALID_ARG;
  if (layout == RA_LAYOUT_ZIGZAG && seqlen % (2 * P) != 0) return RA_ERR_INVALID_ARG;
  return RA_OK;
}

ra_status check_problem(const ra_problem* pr) {
  if (pr == nullptr) return RA_ERR_INVALID_ARG;
  if (pr->batch < 1 || pr->seqlen < 1 || pr->heads < 1 || pr->kv_heads < 1 || pr->P < 1)
    return RA_ERR_INVALID_ARG;
  if (pr->seqlen >= (1 << 30) || pr->P > pr->seqlen || pr->seqlen % pr->P != 0)
    return RA_ERR_INVALID_ARG;
  if (pr->heads % pr->kv_heads != 0) return RA_ERR_INVALID_ARG;
  if (pr->causal != 0 && pr->causal != 1) return RA_ERR_INVALID_ARG;
  if (pr->layout != RA_LAYOUT_CONTIGUOUS && pr->layout != RA_LAYOUT_STRIPED &&
      pr->layout != RA_LAYOUT_ZIGZAG)
    return RA_ERR_INVALID_ARG;
  if (pr->layout == RA_LAYOUT_ZIGZAG && pr->seqlen % (2 * pr->P) != 0) return RA_ERR_INVALID_ARG;
  if (!(pr->scale >= 0.f) || isinf(pr->scale)) return RA_ERR_INVALID_ARG;
  if (pr->o_dtype != RA_DTYPE_BF16 && pr->o_dtype != RA_DTYPE_F32) return RA_ERR_INVALID_ARG;
  if (pr->head_dim != 64 && pr->head_dim != 128) return RA_ERR_UNSUPPORTED;
  // every tensor's element count must fit the kernels' 64-bit offsets and the
  // tensor-map extents (< 2^32 per dimension)
  const double elems = static_cast<double>(pr->batch) * pr->seqlen * pr->heads * pr->head_dim;
  if (elems > 9.0e15) return RA_ERR_INVALID_ARG;
  // the forward launches at most one CTA per (batch, query head, chunk, 128-row
  // query tile); its 1-D grid must stay below 2^31
  const int64_t X = pr->layout == RA_LAYOUT_ZIGZAG ? 2 * pr->P : pr->P;
  const int64_t L = pr->seqlen / X;
  if (static_cast<int64_t>(pr->batch) * pr->heads * X * ((L + 127) / 128) >=
      (static_cast<int64_t>(1) << 31))
    return RA_ERR_UNSUPPORTED;
  return RA_OK;
}

void fill_params(const ra_problem* pr, RingParams* p) {
  memset(p, 0, sizeof(*p));
  p->B = pr->batch;
  p->N = pr->seqlen;
  p->H = pr->heads;
  p->G = pr->kv_heads;
  p->D = pr->head_dim;
  p->P = pr->P;
  p->S = pr->seqlen / pr->P;
  p->layout = pr->layout;
  p->causal = pr->causal;
  p->o_f32 = pr->o_dtype == RA_DTYPE_F32 ? 1 : 0;
  const int hpg = p->H / p->G;
  p->pair_heads = (hpg % 2 == 0) ? 1 : 0;
  p->X = p->layout == kZigzag ? 2 * p->P : p->P;
  p->L = p->layout == kZigzag ? p->S / 2 : p->S;
  p->nq = (p->L + 127) / 128;
  if (p->pair_heads) {
    p->pairs_per_g = hpg / 2;
    p->nqq = p->nq;
  } else {
    p->pairs_per_g = hpg;
    p->nqq = (p->nq + 1) / 2;
  }
  p->units_per_bg = p->pairs_per_g * p->X * p->nqq;
  const double sc = pr->scale > 0.f ? static_cast<double>(pr->scale) : 1.0 / sqrt(static_cast<double>(p->D));
  p->scale = static_cast<float>(sc);
  p->scale_log2 = static_cast<float>(sc * 1.4426950408889634);
  p->timeout_ns = g_wait_limit_ns.load();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Tensor map over a [B, N, heads, D] bf16 tensor seen as 5-D (innermost first):
// contiguous (D, heads, S, P, B) — token = u*S + i; striped (D, heads, P, S, B) —
// token = i*P + u. A box is 64 columns of one head over box_rows local rows of
// one shard, written to shared memory with the 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* base, int B, int N, int heads, int D, int S, int P,
                 int layout, int box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t tok = static_cast<cuuint64_t>(heads) * D * 2;
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5];
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  dims[0] = D;
  dims[1] = heads;
  box[0] = 64;
  box[1] = 1;
  strides[0] = static_cast<cuuint64_t>(D) * 2;
  if (layout == kContiguous) {
    dims[2] = S;
    dims[3] = P;
    strides[1] = tok;
    strides[2] = tok * S;
    box[2] = static_cast<cuuint32_t>(box_rows);
    box[3] = 1;
  } else {
    dims[2] = P;
    dims[3] = S;
    strides[1] = tok;
    strides[2] = tok * P;
    box[2] = 1;
    box[3] = static_cast<cuuint32_t>(box_rows);
  }
  dims[4] = B;
  strides[3] = tok * N;
  box[4] = 1;
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

ra_status launch_result(cudaError_t e) { return e == cudaSuccess ? RA_OK : cuda_failed(e); }

ra_status run_tc(const RingParams& p, cudaStream_t st) {
  // zigzag tiles by chunk: the contiguous view with X = 2P chunks of L = S/2 tokens
  const int ml = p.layout == kZigzag ? kContiguous : p.layout;
  CUtensorMap tq, tk, tv;
  if (!encode_rows(&tq, p.q, p.B, p.N, p.H, p.D, p.L, p.X, ml) ||
      !encode_rows(&tk, p.k, p.B, p.N, p.G, p.D, p.L, p.X, ml) ||
      !encode_rows(&tv, p.v, p.B, p.N, p.G, p.D, p.L, p.X, ml))
    return cuda_failed(cudaErrorInvalidValue);
  return launch_result(launch_ring_tc(p, tq, tk, tv, st));
}

ra_status check_step_args(const ra_problem* pr, int32_t s, const void* q, const void* k,
                          const void* v, float* m, float* z, float* y) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  if (s < 0 || s >= pr->P) return RA_ERR_INVALID_ARG;
  if (!q || !k || !v || !m || !z || !y) return RA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(m) || !aligned16(z) ||
      !aligned16(y))
    return RA_ERR_INVALID_ARG;
  const Bytes b = tensor_bytes(pr);
  if (!writes_disjoint({{m, b.rows}, {z, b.rows}, {y, b.y}}, {{q, b.q}, {k, b.kv}, {v, b.kv}}))
    return RA_ERR_INVALID_ARG;
  return RA_OK;
}

// Number of partials the decode phase writes (one per shard segment and key chunk).
int64_t decode_parts(const ra_problem* pr) {
  return ra::decode_parts(pr->seqlen / pr->P, pr->P, pr->layout);
}

size_t decode_workspace(const ra_problem* pr, int32_t n_q) {
  const size_t parts = static_cast<size_t>(decode_parts(pr));
  const size_t rows = static_cast<size_t>(pr->batch) * pr->heads * n_q;
  return parts * rows * (static_cast<size_t>(pr->head_dim) + 1) * sizeof(float);
}

// Backward workspace, per (batch, head, chunk, 128-row query tile): 1 KiB of
// statistics plus two 4 KiB extension tiles; then one 4 KiB key-side tile.
int64_t bwd_tiles(const ra_problem* pr) {
  const int S = pr->seqlen / pr->P;
  const int X = pr->layout == RA_LAYOUT_ZIGZAG ? 2 * pr->P : pr->P;
  const int L = pr->layout == RA_LAYOUT_ZIGZAG ? S / 2 : S;
  return static_cast<int64_t>(pr->batch) * pr->heads * X * ((L + 127) / 128);
}
size_t bwd_workspace(const ra_problem* pr) {
  return static_cast<size_t>(bwd_tiles(pr)) * (1024 + 2 * 4096) + 4096;
}

// 2-D map over the extension rows (16 bf16 each), boxes of 128 rows, 32-byte swizzle.
bool encode_ext(CUtensorMap* m, const void* base, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {16, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {32};
  const cuuint32_t box[2] = {16, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device slot of ring_attn_fwd_host: one piece — one sequence's query heads of
// one kv group and that kv head — as contiguous q, k, v, o, lse, each rounded up
// to 256 bytes.
struct HostSlot {
  size_t q, kv, o, lse, total;
};
HostSlot host_slot(const ra_problem* pr) {
  auto r256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t hpg = static_cast<size_t>(pr->heads / pr->kv_heads);
  HostSlot s;
  s.q = r256(static_cast<size_t>(pr->seqlen) * hpg * pr->head_dim * 2);
  s.kv = r256(static_cast<size_t>(pr->seqlen) * pr->head_dim * 2);
  s.o = r256(static_cast<size_t>(pr->seqlen) * hpg * pr->head_dim *
             (pr->o_dtype == RA_DTYPE_F32 ? 4 : 2));
  s.lse = r256(hpg * pr->seqlen * sizeof(float));
  s.total = s.q + 2 * s.kv + s.o + s.lse;
  return s;
}
// Device slots of ring_attn_fwd_host: at least 2 (or one per piece if fewer) are
// required; the recommended workspace holds kHostSlots (or one per piece), so the input
// copies can run up to kHostSlots - 1 pieces ahead of the kernels and absorb copies
// that stall (tens of milliseconds at a time were seen on the host link).
constexpr int64_t kHostSlots = 16;
int64_t host_pieces(const ra_problem* pr) {
  return static_cast<int64_t>(pr->batch) * pr->kv_heads;
}
typedef CUresult (*PointerAttrFn)(void*, CUpointer_attribute, CUdeviceptr);

PointerAttrFn pointer_attr_fn() {
  static PointerAttrFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PointerAttrFn>(ptr);
  });
  return fn;
}

// True when [p, p + bytes) is page-locked host memory that this device reaches at the
// same address, so that kernels may read or write it directly: its first and last
// byte are such memory, and one allocation (or registration) holds the whole range,
// so no byte between them is unmapped. False for pageable memory, for ranges that
// run over the end of their allocation, and whenever a query fails (the copy engines
// then move the tensor).
bool mapped_host(const void* p, size_t bytes) {
  if (bytes == 0 || (reinterpret_cast<uintptr_t>(p) & 3u)) return false;
  const char* ends[2] = {static_cast<const char*>(p), static_cast<const char*>(p) + bytes - 1};
  for (const char* e : ends) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, e) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer != static_cast<const void*>(e))
      return false;
  }
  PointerAttrFn fn = pointer_attr_fn();
  if (fn == nullptr) return false;
  CUdeviceptr start = 0;
  size_t size = 0;
  const CUdeviceptr at = static_cast<CUdeviceptr>(reinterpret_cast<uintptr_t>(p));
  if (fn(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, at) != CUDA_SUCCESS ||
      fn(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, at) != CUDA_SUCCESS)
    return false;
  return at >= start && at - start <= size && bytes <= size - (at - start);
}

size_t fwd_host_min_workspace(const ra_problem* pr) {
  const int64_t n = host_pieces(pr);
  return host_slot(pr).total * static_cast<size_t>(n < 2 ? n : 2);
}
size_t fwd_host_workspace(const ra_problem* pr) {
  const int64_t n = host_pieces(pr);
  return host_slot(pr).total * static_cast<size_t>(n < kHostSlots ? n : kHostSlots);
}

}  // namespace

extern "C" {

ra_status ring_attn_fwd(const ra_problem* pr, const void* q, const void* k, const void* v,
                        void* o, float* lse, void* stream) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  if (!q || !k || !v || !o || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return RA_ERR_INVALID_ARG;
  const Bytes b = tensor_bytes(pr);
  if (!writes_disjoint({{o, b.o}, {lse, b.rows}}, {{q, b.q}, {k, b.kv}, {v, b.kv}}))
    return RA_ERR_INVALID_ARG;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {q, k, v, o, lse})) != RA_OK) return st;
  RingParams p;
  fill_params(pr, &p);
  p.s_begin = 0;
  p.s_end = p.P;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.status = d->status;
  return run_tc(p, static_cast<cudaStream_t>(stream));
}

size_t ring_attn_fwd_host_workspace_bytes(const ra_problem* pr) {
  if (check_problem(pr) != RA_OK) return 0;
  return fwd_host_workspace(pr);
}

ra_status ring_attn_fwd_host(const ra_problem* pr, const void* q, const void* k, const void* v,
                             void* o, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream, void* copy_stream) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  if (!q || !k || !v || !o || !lse || !workspace || !aligned16(workspace))
    return RA_ERR_INVALID_ARG;
  if (workspace_bytes < fwd_host_min_workspace(pr)) return RA_ERR_INVALID_ARG;
  {
    const Bytes b = tensor_bytes(pr);
    if (!writes_disjoint({{o, b.o}, {lse, b.rows}, {workspace, workspace_bytes}},
                         {{q, b.q}, {k, b.kv}, {v, b.kv}}))
      return RA_ERR_INVALID_ARG;
  }
  if (host_pieces(pr) > (1 << 24)) return RA_ERR_UNSUPPORTED;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {workspace})) != RA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);        // kernels
  const HostSlot hs = host_slot(pr);
  const int B = pr->batch, G = pr->kv_heads, H = pr->heads, N = pr->seqlen, D = pr->head_dim;
  const int hpg = H / G;
  const int n = static_cast<int>(host_pieces(pr));
  const int64_t fit = static_cast<int64_t>(workspace_bytes / hs.total);
  const int S = static_cast<int>(fit < n ? fit : n);                // device slots in use
  // A piece (b, g) is the ring forward of sequence b restricted to kv group g:
  // its query heads [g hpg, (g+1) hpg) against kv head g, a problem of its own.
  ra_problem one = *pr;
  one.batch = 1;
  one.heads = hpg;
  one.kv_heads = 1;
  RingParams p;
  fill_params(&one, &p);
  p.s_begin = 0;
  p.s_end = p.P;
  p.status = d->status;
  const size_t row_q = static_cast<size_t>(H) * D * 2;      // bytes per token of q
  const size_t row_kv = static_cast<size_t>(G) * D * 2;     // bytes per token of k, v
  const size_t w_q = static_cast<size_t>(hpg) * D * 2;      // a piece's bytes per token
  const size_t o_elem = pr->o_dtype == RA_DTYPE_F32 ? 4 : 2;
  const size_t row_o = static_cast<size_t>(H) * D * o_elem;  // the same for o
  const size_t w_o = static_cast<size_t>(hpg) * D * o_elem;
  const size_t w_kv = static_cast<size_t>(D) * 2;
  const size_t lse_piece = static_cast<size_t>(hpg) * N * sizeof(float);
  // Tensors in page-locked memory mapped at the same address are moved by copy kernels
  // (hostcopy.cu); the rest by the copy engines.
  const size_t bq = static_cast<size_t>(B) * N * row_q, bkv = static_cast<size_t>(B) * N * row_kv;
  const bool zq = mapped_host(q, bq), zk = mapped_host(k, bkv), zv = mapped_host(v, bkv);
  const bool zo = mapped_host(o, static_cast<size_t>(B) * N * row_o), zl = mapped_host(lse, static_cast<size_t>(B) * G * lse_piece);
  // Outputs leave on a stream of this call's own, so a stalled output copy never holds
  // up the inputs (and the reverse); inputs come in on another stream of its own when
  // copy kernels move any of them, else on copy_stream. Streams of copy kernels run at
  // the device's highest priority, so their blocks go ahead of the ring kernel's.
  int lo_prio = 0, hi_prio = 0;
  cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo_prio, &hi_prio);
  if (e != cudaSuccess) return cuda_failed(e);
  cudaStream_t os = nullptr, own_is = nullptr;
  e = cudaStreamCreateWithPriority(&os, cudaStreamNonBlocking, hi_prio);
  if (e != cudaSuccess) return cuda_failed(e);
  if (zq || zk || zv) {
    e = cudaStreamCreateWithPriority(&own_is, cudaStreamNonBlocking, hi_prio);
    if (e != cudaSuccess) {
      cudaStreamDestroy(os);
      return cuda_failed(e);
    }
  }
  const cudaStream_t is = own_is ? own_is : static_cast<cudaStream_t>(copy_stream);
  // events: start, inputs-done joined back, end; per piece: inputs in, kernel done, outputs out
  const int n_ev = 3 + 3 * n;
  cudaEvent_t* ev = new (std::nothrow) cudaEvent_t[n_ev];
  if (ev == nullptr) {
    cudaStreamDestroy(os);
    if (own_is) cudaStreamDestroy(own_is);
    return cuda_failed(cudaErrorMemoryAllocation);
  }
  int made = 0;
  for (; made < n_ev && e == cudaSuccess; ++made)
    e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
  if (e != cudaSuccess) --made;
  const cudaEvent_t ev_start = ev[0], ev_in_end = ev[1], ev_end = ev[2];
  auto ev_in = [&](int i) { return ev[3 + i]; };
  auto ev_k = [&](int i) { return ev[3 + n + i]; };
  auto ev_out = [&](int i) { return ev[3 + 2 * n + i]; };
  auto slot = [&](int i) { return static_cast<uint8_t*>(workspace) + (i % S) * hs.total; };
  // Copy kernels run 38 blocks (a quarter of the SMs) while ring kernels share the GPU:
  // they have slack and fewer blocks take fewer SM slots from the ring kernel; four
  // blocks per SM when the first piece's inputs or the last piece's outputs move with
  // nothing else running.
  constexpr int kCopyBlocks = 38, kCopyBlocksAlone = 4 * 152;
  auto h2d = [&](int i) -> cudaError_t {
    const int b = i / G, g = i % G;
    const int blocks = i == 0 ? kCopyBlocksAlone : kCopyBlocks;
    uint8_t* s0 = slot(i);
    const uint8_t* qs = static_cast<const uint8_t*>(q) + static_cast<size_t>(b) * N * row_q + g * w_q;
    const uint8_t* ks = static_cast<const uint8_t*>(k) + static_cast<size_t>(b) * N * row_kv + g * w_kv;
    const uint8_t* vs = static_cast<const uint8_t*>(v) + static_cast<size_t>(b) * N * row_kv + g * w_kv;
    auto in = [&](bool kernel, void* dst, const void* src, size_t pitch, size_t width) {
      return kernel ? launch_rows_copy(dst, width, src, pitch, width, N, blocks, is)
                    : cudaMemcpy2DAsync(dst, width, src, pitch, width, N, cudaMemcpyHostToDevice, is);
    };
    cudaError_t r = in(zq, s0, qs, row_q, w_q);
    if (r == cudaSuccess) r = in(zk, s0 + hs.q, ks, row_kv, w_kv);
    if (r == cudaSuccess) r = in(zv, s0 + hs.q + hs.kv, vs, row_kv, w_kv);
    if (r == cudaSuccess) r = cudaEventRecord(ev_in(i), is);
    return r;
  };
  if (e == cudaSuccess) e = cudaEventRecord(ev_start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(is, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(os, ev_start, 0);
  for (int i = 0; i < S && e == cudaSuccess; ++i) e = h2d(i);        // fill every slot
  for (int i = 0; i < n && e == cudaSuccess; ++i) {
    const int b = i / G, g = i % G;
    uint8_t* s0 = slot(i);
    e = cudaStreamWaitEvent(cs, ev_in(i), 0);
    if (e != cudaSuccess) break;
    p.q = s0;
    p.k = s0 + hs.q;
    p.v = s0 + hs.q + hs.kv;
    p.o = s0 + hs.q + 2 * hs.kv;
    p.lse = reinterpret_cast<float*>(s0 + hs.q + 2 * hs.kv + hs.o);
    if ((st = run_tc(p, cs)) != RA_OK) break;
    e = cudaEventRecord(ev_k(i), cs);
    // outputs of piece i out once its kernel is done
    if (e == cudaSuccess) e = cudaStreamWaitEvent(os, ev_k(i), 0);
    uint8_t* od = static_cast<uint8_t*>(o) + static_cast<size_t>(b) * N * row_o + g * w_o;
    // lse [B, H, N]: the group's heads are consecutive rows
    uint8_t* ld = reinterpret_cast<uint8_t*>(lse) + (static_cast<size_t>(b) * G + g) * lse_piece;
    const int oblocks = i + 1 == n ? kCopyBlocksAlone : kCopyBlocks;
    if (e == cudaSuccess)
      e = zo ? launch_rows_copy(od, row_o, p.o, w_o, w_o, N, oblocks, os)
             : cudaMemcpy2DAsync(od, row_o, p.o, w_o, w_o, N, cudaMemcpyDeviceToHost, os);
    if (e == cudaSuccess)
      e = zl ? launch_rows_copy(ld, lse_piece, p.lse, lse_piece, lse_piece, 1, oblocks, os)
             : cudaMemcpyAsync(ld, p.lse, lse_piece, cudaMemcpyDeviceToHost, os);
    if (e == cudaSuccess) e = cudaEventRecord(ev_out(i), os);
    // the slot is free once its outputs are out (its inputs were consumed before):
    // the inputs of piece i + S come in there
    if (e == cudaSuccess && i + S < n) e = cudaStreamWaitEvent(is, ev_out(i), 0);
    if (e == cudaSuccess && i + S < n) e = h2d(i + S);
  }
  // Join both copy streams back into `stream`, also after an error: copies already
  // queued may still write the workspace, and the caller orders its reuse on `stream`.
  if (made == n_ev) {
    cudaError_t j = cudaEventRecord(ev_in_end, is);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(cs, ev_in_end, 0);
    if (j == cudaSuccess) j = cudaEventRecord(ev_end, os);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(cs, ev_end, 0);
    if (e == cudaSuccess) e = j;
  }
  for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);   // released once they complete
  delete[] ev;
  cudaStreamDestroy(os);                                      // likewise
  if (own_is) cudaStreamDestroy(own_is);
  if (st != RA_OK) return st;
  return e == cudaSuccess ? RA_OK : cuda_failed(e);
}

int32_t ring_attn_host_mapped(const void* p, size_t bytes) {
  DevInfo* d = nullptr;
  if (p == nullptr || current_device(&d) != RA_OK) return 0;
  return mapped_host(p, bytes) ? 1 : 0;
}

ra_status ring_attn_step(const ra_problem* pr, int32_t s, int32_t first, const void* q,
                         const void* k, const void* v, float* m, float* z, float* y,
                         void* stream) {
  ra_status st = check_step_args(pr, s, q, k, v, m, z, y);
  if (st != RA_OK) return st;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {q, k, v, m, z, y})) != RA_OK) return st;
  RingParams p;
  fill_params(pr, &p);
  p.s_begin = s;
  p.s_end = s + 1;
  p.step_mode = 1;
  p.load_state = first ? 0 : 1;
  p.q = q;
  p.k = k;
  p.v = v;
  p.m = m;
  p.z = z;
  p.y = y;
  p.status = d->status;
  return run_tc(p, static_cast<cudaStream_t>(stream));
}

ra_status ring_attn_step_simt(const ra_problem* pr, int32_t s, int32_t first, const void* q,
                              const void* k, const void* v, float* m, float* z, float* y,
                              void* stream) {
  ra_status st = check_step_args(pr, s, q, k, v, m, z, y);
  if (st != RA_OK) return st;
  if (static_cast<long long>(pr->batch) * pr->heads > 65535 || pr->P > 65535)
    return RA_ERR_UNSUPPORTED;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {q, k, v, m, z, y})) != RA_OK) return st;
  RingParams p;
  fill_params(pr, &p);
  p.s_begin = s;
  p.s_end = s + 1;
  p.step_mode = 1;
  p.load_state = first ? 0 : 1;
  p.q = q;
  p.k = k;
  p.v = v;
  p.m = m;
  p.z = z;
  p.y = y;
  p.status = d->status;
  return launch_result(launch_ring_simt(p, static_cast<cudaStream_t>(stream)));
}

ra_status ring_attn_finalize(const ra_problem* pr, const float* m, const float* z,
                             const float* y, void* o, float* lse, void* stream) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  if (!m || !z || !y || !o || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned16(m) || !aligned16(z) || !aligned16(y) || !aligned16(o) || !aligned16(lse))
    return RA_ERR_INVALID_ARG;
  const Bytes b = tensor_bytes(pr);
  if (!writes_disjoint({{o, b.o}, {lse, b.rows}}, {{m, b.rows}, {z, b.rows}, {y, b.y}}))
    return RA_ERR_INVALID_ARG;
  if (static_cast<long long>(pr->batch) > 65535 || pr->heads > 65535) return RA_ERR_UNSUPPORTED;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {m, z, y, o, lse})) != RA_OK) return st;
  RingParams p;
  fill_params(pr, &p);
  p.m = const_cast<float*>(m);
  p.z = const_cast<float*>(z);
  p.y = const_cast<float*>(y);
  p.o = o;
  p.lse = lse;
  p.status = d->status;
  return launch_result(launch_finalize(p, static_cast<cudaStream_t>(stream)));
}

ra_status ring_attn_merge(int32_t n_parts, int32_t batch, int32_t seqlen, int32_t heads,
                          int32_t head_dim, const float* o_parts, const float* lse_parts,
                          void* o, float* lse, void* stream) {
  if (n_parts < 1 || n_parts > 1024 || batch < 1 || seqlen < 1 || heads < 1)
    return RA_ERR_INVALID_ARG;
  if (batch > 65535 || heads > 65535) return RA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return RA_ERR_UNSUPPORTED;
  if (!o_parts || !lse_parts || !o || !lse) return RA_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o) || !aligned16(lse))
    return RA_ERR_INVALID_ARG;
  {
    const size_t rows = static_cast<size_t>(batch) * seqlen * heads;
    const size_t n = static_cast<size_t>(n_parts);
    if (!writes_disjoint({{o, rows * head_dim * 2}, {lse, rows * sizeof(float)}},
                         {{o_parts, n * rows * head_dim * sizeof(float)},
                          {lse_parts, n * rows * sizeof(float)}}))
      return RA_ERR_INVALID_ARG;
  }
  DevInfo* d = nullptr;
  ra_status st = current_device(&d);
  if (st != RA_OK) return st;
  if ((st = resident(d, {o_parts, lse_parts, o, lse})) != RA_OK) return st;
  return launch_result(launch_merge(n_parts, batch, seqlen, heads, head_dim, o_parts, lse_parts,
                                    o, false, lse, static_cast<cudaStream_t>(stream)));
}

ra_status ring_attn_shard_map(int32_t layout, int32_t seqlen, int32_t P, int32_t* owner,
                              int32_t* local, int32_t* token_of) {
  if (check_layout_sizes(layout, seqlen, P) != RA_OK) return RA_ERR_INVALID_ARG;
  if (!owner || !local || !token_of) return RA_ERR_INVALID_ARG;
  const int32_t S = seqlen / P;
  for (int32_t t = 0; t < seqlen; ++t) {
    owner[t] = owner_of(layout, S, P, t);
    local[t] = local_of(layout, S, P, t);
    token_of[t] = pos_of(layout, S, P, t / S, t % S);
  }
  return RA_OK;
}

ra_status ring_attn_shard_map_device(int32_t layout, int32_t seqlen, int32_t P, int32_t* owner,
                                     int32_t* local, int32_t* token_of, void* stream) {
  if (check_layout_sizes(layout, seqlen, P) != RA_OK) return RA_ERR_INVALID_ARG;
  if (!owner || !local || !token_of) return RA_ERR_INVALID_ARG;
  DevInfo* d = nullptr;
  ra_status st = current_device(&d);
  if (st != RA_OK) return st;
  if ((st = resident(d, {owner, local, token_of})) != RA_OK) return st;
  return launch_result(
      launch_shard_map(layout, seqlen, P, owner, local, token_of, static_cast<cudaStream_t>(stream)));
}

ra_status ring_attn_tile_classes(const ra_problem* pr, int32_t u, int32_t b, int8_t* classes,
                                 void* stream) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  if (u < 0 || u >= pr->P || b < 0 || b >= pr->P || classes == nullptr) return RA_ERR_INVALID_ARG;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {classes})) != RA_OK) return st;
  RingParams p;
  fill_params(pr, &p);
  return launch_result(launch_tile_classes(p, u, b, classes, static_cast<cudaStream_t>(stream)));
}

ra_status ring_attn_mask(const ra_problem* pr, int32_t u, int32_t b, uint8_t* mask,
                         void* stream) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  if (u < 0 || u >= pr->P || b < 0 || b >= pr->P || mask == nullptr) return RA_ERR_INVALID_ARG;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {mask})) != RA_OK) return st;
  RingParams p;
  fill_params(pr, &p);
  return launch_result(launch_mask(p, u, b, mask, static_cast<cudaStream_t>(stream)));
}

size_t ring_attn_decode_workspace_bytes(const ra_problem* pr, int32_t n_q) {
  if (check_problem(pr) != RA_OK || n_q < 1) return 0;
  return decode_workspace(pr, n_q);
}

size_t ring_attn_bwd_workspace_bytes(const ra_problem* pr) {
  if (check_problem(pr) != RA_OK) return 0;
  return bwd_workspace(pr);
}

ra_status ring_attn_bwd(const ra_problem* pr, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout, void* dq, void* dk,
                        void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  const void* in[] = {q, k, v, o, lse, dout, dq, dk, dv, workspace};
  for (const void* ptr : in)
    if (ptr == nullptr || !aligned16(ptr)) return RA_ERR_INVALID_ARG;
  if (workspace_bytes < bwd_workspace(pr)) return RA_ERR_INVALID_ARG;
  {
    const Bytes b = tensor_bytes(pr);
    if (!writes_disjoint({{dq, b.q}, {dk, b.kv}, {dv, b.kv}, {workspace, bwd_workspace(pr)}},
                         {{q, b.q}, {k, b.kv}, {v, b.kv}, {o, b.o}, {lse, b.rows}, {dout, b.q}}))
      return RA_ERR_INVALID_ARG;
  }
  // the extension rows are addressed by 32-bit TMA coordinates
  if (bwd_tiles(pr) * 2 * 128 + 128 >= (static_cast<int64_t>(1) << 31)) return RA_ERR_UNSUPPORTED;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {q, k, v, o, lse, dout, dq, dk, dv, workspace})) != RA_OK) return st;
  RingParams f;
  fill_params(pr, &f);
  BwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = f.B;
  p.N = f.N;
  p.H = f.H;
  p.G = f.G;
  p.D = f.D;
  p.S = f.S;
  p.P = f.P;
  p.layout = f.layout;
  p.causal = f.causal;
  p.X = f.X;
  p.L = f.L;
  p.nt = f.nq;
  p.tiles = static_cast<int32_t>(bwd_tiles(pr));
  p.o_f32 = f.o_f32;
  p.scale = f.scale;
  p.scale_log2 = f.scale_log2;
  p.timeout_ns = f.timeout_ns;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.ws = static_cast<float*>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = d->status;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // zigzag tiles by chunk: the contiguous view with X = 2P chunks of L = S/2 tokens
  const int ml = p.layout == kZigzag ? kContiguous : p.layout;
  CUtensorMap tq, tdo, tk, tv, text;
  const void* ext = static_cast<const uint8_t*>(workspace) + static_cast<size_t>(p.tiles) * 1024;
  if (!encode_rows(&tq, q, p.B, p.N, p.H, p.D, p.L, p.X, ml) ||
      !encode_rows(&tdo, dout, p.B, p.N, p.H, p.D, p.L, p.X, ml) ||
      !encode_rows(&tk, k, p.B, p.N, p.G, p.D, p.L, p.X, ml) ||
      !encode_rows(&tv, v, p.B, p.N, p.G, p.D, p.L, p.X, ml) ||
      !encode_ext(&text, ext, static_cast<int64_t>(p.tiles) * 2 * 128 + 128))
    return cuda_failed(cudaErrorInvalidValue);
  if ((st = launch_result(launch_bwd_prep(p, s))) != RA_OK) return st;
  if ((st = launch_result(launch_bwd_dkdv(p, tq, tdo, tk, tv, text, s))) != RA_OK) return st;
  return launch_result(launch_bwd_dq(p, tq, tdo, tk, tv, s));
}

ra_status ring_attn_decode(const ra_problem* pr, int32_t n_q, int32_t q_pos0, const void* q,
                           const void* k, const void* v, void* o, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream) {
  ra_status st = check_problem(pr);
  if (st != RA_OK) return st;
  if (n_q < 1 || n_q > 4096 || q_pos0 < 0) return RA_ERR_INVALID_ARG;
  if (pr->causal && static_cast<int64_t>(q_pos0) + n_q > pr->seqlen) return RA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse || !workspace) return RA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return RA_ERR_INVALID_ARG;
  if (workspace_bytes < decode_workspace(pr, n_q)) return RA_ERR_INVALID_ARG;
  {
    const Bytes b = tensor_bytes(pr);
    const size_t qrows = static_cast<size_t>(pr->batch) * n_q * pr->heads;
    const size_t o_elem = pr->o_dtype == RA_DTYPE_F32 ? 4 : 2;
    if (!writes_disjoint({{o, qrows * pr->head_dim * o_elem}, {lse, qrows * sizeof(float)},
                          {workspace, decode_workspace(pr, n_q)}},
                         {{q, qrows * pr->head_dim * 2}, {k, b.kv}, {v, b.kv}}))
      return RA_ERR_INVALID_ARG;
  }
  const int64_t parts = decode_parts(pr);
  // launch limits of the partial phase (grid z = batch * P) and of the merge
  if (parts > 1024 || static_cast<int64_t>(pr->batch) * pr->P > 65535 || pr->batch > 65535 ||
      pr->heads > 65535)
    return RA_ERR_UNSUPPORTED;
  DevInfo* d = nullptr;
  if ((st = current_device(&d)) != RA_OK) return st;
  if ((st = resident(d, {q, k, v, o, lse, workspace})) != RA_OK) return st;
  RingParams p;
  fill_params(pr, &p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.status = d->status;
  float* o_parts = static_cast<float*>(workspace);
  float* lse_parts = o_parts + static_cast<size_t>(parts) * pr->batch * n_q * pr->heads * pr->head_dim;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // K/V tiles of 32 keys; zigzag tiles by chunk: the contiguous view over 2P chunks
  const int ml = p.layout == kZigzag ? kContiguous : p.layout;
  CUtensorMap tk, tv;
  if (!encode_rows(&tk, k, p.B, p.N, p.G, p.D, p.L, p.X, ml, 32) ||
      !encode_rows(&tv, v, p.B, p.N, p.G, p.D, p.L, p.X, ml, 32))
    return cuda_failed(cudaErrorInvalidValue);
  p.o = o;
  p.lse = lse;
  const bool clustered = decode_clustered(p, n_q);
  cudaError_t e = launch_decode_partials(p, tk, tv, n_q, q_pos0, o_parts, lse_parts, clustered, cs);
  if (e != cudaSuccess) return cuda_failed(e);
  if (clustered) return RA_OK;
  return launch_result(launch_merge(static_cast<int>(parts), pr->batch, n_q, pr->heads,
                                    pr->head_dim, o_parts, lse_parts, o, p.o_f32 != 0, lse,
                                    cs));
}

ra_status ring_attn_last_error(int32_t* device_code) {
  if (device_code == nullptr) return RA_ERR_INVALID_ARG;
  DevInfo* d = nullptr;
  ra_status st = current_device(&d);
  if (st != RA_OK) return st;
  int code = 0;
  const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&code, g_status, sizeof(int));
  if (e != cudaSuccess) return cuda_failed(e);
  if ((e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int))) != cudaSuccess) return cuda_failed(e);
  *device_code = code;
  return RA_OK;
}

ra_status ring_attn_selftest_wait_limit(uint64_t limit_ns) {
  if (limit_ns > kWaitLimitNs) return RA_ERR_INVALID_ARG;
  g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : limit_ns);
  return RA_OK;
}

ra_status ring_attn_selftest_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return RA_ERR_INVALID_ARG;
  DevInfo* d = nullptr;
  ra_status st = current_device(&d);
  if (st != RA_OK) return st;
  return launch_result(launch_selftest_timeout(limit_ns, d->status, static_cast<cudaStream_t>(stream)));
}

int32_t ring_attn_last_cuda_error(void) { return g_last_cuda_error; }

const char* ring_attn_cuda_error_name(int32_t code) {
  return cudaGetErrorName(static_cast<cudaError_t>(code));
}

const char* ra_status_str(ra_status s) {
  switch (s) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_TIMEOUT: return "RA_ERR_TIMEOUT";
    case RA_ERR_BOUNDS: return "RA_ERR_BOUNDS";
  }
  return "RA_ERR_UNKNOWN";
}

int32_t ring_attn_version(void) { return 102; }

int32_t ring_attn_debug_checks(void) { return kDebugChecks ? 1 : 0; }

ra_status ring_attn_selftest_bounds(void* stream) {
  DevInfo* d = nullptr;
  ra_status st = current_device(&d);
  if (st != RA_OK) return st;
  return launch_result(launch_selftest_bounds(d->status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
