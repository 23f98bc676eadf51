// C ABI of libkaio_qkv: argument validation, device checks and dispatch to
// the kernels. No computation happens on
// the host: every output element is produced by a kernel on the device.
//
// The validation mirrors the input contract of the direct-call bridge on
// "kaio-candle -- src/qkv_project_int4.rs" (qkv_project_int4: K a multiple of
// the locked group size 128, packed rows K/8, scale rows K/128, one N shared by
// the six weight/scale tensors, all inputs on the one device, dimensions
// within u32) and of MatmulTcAsyncOp::cuda_fwd on
// "kaio-candle 0.2.0 -- src/matmul_tc_async.rs" (inner dimensions match, no CPU
// fallback). Shapes are implied here by (M, N, K), so a row-count mismatch
// cannot be expressed; what remains checkable is checked.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/kaio_qkv.h"
#include "kaio_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(KAIO_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceInfo {
  int major = 0, minor = 0, sms = 0;
  bool ok = false;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;

// Current device; fills `info` (cached, per host thread after the first
// lookup). Returns KAIO_OK or an error status.
int current_device(int* dev, DeviceInfo* info) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  constexpr int kSlots = 64;
  thread_local DeviceInfo slots[kSlots];
  thread_local bool filled[kSlots] = {};
  if (*dev >= 0 && *dev < kSlots && filled[*dev]) {
    *info = slots[*dev];
  } else {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_devices.find(*dev);
    if (it == g_devices.end()) {
      DeviceInfo d;
      if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
      d.ok = (d.major == 10 && d.minor == 3);
      it = g_devices.emplace(*dev, d).first;
    }
    *info = it->second;
    if (*dev >= 0 && *dev < kSlots) {
      slots[*dev] = *info;
      filled[*dev] = true;
    }
  }
  if (!info->ok)
    return fail(KAIO_ERR_UNSUPPORTED_DEVICE,
                "device %d has compute capability %d.%d; this library is built for sm_103a "
                "(compute capability 10.3, GB300) only",
                *dev, info->major, info->minor);
  return KAIO_OK;
}

#define KAIO_TRY_FN(expr)        \
  do {                           \
    const int st__ = (expr);     \
    if (st__ != KAIO_OK) return st__; \
  } while (0)

struct Span {
  const char* name;
  const void* p;
  size_t bytes;
};

int check_not_null(const Span* s, int n) {
  for (int i = 0; i < n; ++i)
    if (s[i].p == nullptr) return fail(KAIO_ERR_INVALID_VALUE, "%s is a null pointer", s[i].name);
  return KAIO_OK;
}

int check_aligned(const Span* s, int n) {
  for (int i = 0; i < n; ++i)
    if (reinterpret_cast<uintptr_t>(s[i].p) % 16 != 0)
      return fail(KAIO_ERR_MISALIGNED, "%s (%p) is not 16-byte aligned", s[i].name, s[i].p);
  return KAIO_OK;
}

bool overlaps(const Span& a, const Span& b) {
  if (a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Every output must be disjoint from every input and from the other outputs.
int check_overlap(const Span* in, int n_in, const Span* out, int n_out) {
  for (int i = 0; i < n_out; ++i) {
    for (int j = 0; j < n_in; ++j)
      if (overlaps(out[i], in[j]))
        return fail(KAIO_ERR_INVALID_VALUE, "output %s overlaps input %s", out[i].name, in[j].name);
    for (int j = i + 1; j < n_out; ++j)
      if (overlaps(out[i], out[j]))
        return fail(KAIO_ERR_INVALID_VALUE, "outputs %s and %s overlap", out[i].name, out[j].name);
  }
  return KAIO_OK;
}

// Each pointer must be device (or managed) memory of the current device. One
// driver query per allocation: it also returns the allocation's address
// range, and a later tensor lying wholly inside a range already found to be
// device memory of this device needs no query of its own (within this call;
// nothing is remembered across calls, since memory may be freed in between).
// Anything that is not plain device memory, or an unavailable driver entry
// point, takes the runtime query and its messages.
using PointerGetAttributesFn = CUresult (*)(unsigned int, CUpointer_attribute*, void**, CUdeviceptr);

PointerGetAttributesFn pointer_attributes_fn() {
  static PointerGetAttributesFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PointerGetAttributesFn>(f);
  });
  return fn;
}

int check_one_on_device(const Span& s, int dev) {
  cudaPointerAttributes a{};
  cudaError_t e = cudaPointerGetAttributes(&a, s.p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(KAIO_ERR_INVALID_VALUE, "%s (%p) is not CUDA device memory (%s)", s.name, s.p,
                cudaGetErrorName(e));
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return fail(KAIO_ERR_INVALID_VALUE, "%s (%p) is not device memory (memory type %d)", s.name, s.p,
                static_cast<int>(a.type));
  if (a.device != dev)
    return fail(KAIO_ERR_INVALID_VALUE, "%s is on device %d but the current device is %d", s.name,
                a.device, dev);
  return KAIO_OK;
}

int check_on_device(const Span* s, int n, int dev) {
  const PointerGetAttributesFn fn = pointer_attributes_fn();
  constexpr int kMaxRanges = 16;
  uintptr_t lo[kMaxRanges], hi[kMaxRanges];
  int nr = 0;
  for (int i = 0; i < n; ++i) {
    const uintptr_t p0 = reinterpret_cast<uintptr_t>(s[i].p), p1 = p0 + (s[i].bytes ? s[i].bytes : 1);
    bool known = false;
    for (int r = 0; r < nr && !known; ++r) known = p0 >= lo[r] && p1 <= hi[r];
    if (known) continue;
    if (fn) {
      unsigned int mtype = 0;
      int ordinal = -1;
      CUdeviceptr start = 0;
      size_t size = 0;
      CUpointer_attribute attrs[4] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL,
                                      CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, CU_POINTER_ATTRIBUTE_RANGE_SIZE};
      void* data[4] = {&mtype, &ordinal, &start, &size};
      if (fn(4, attrs, data, static_cast<CUdeviceptr>(p0)) == CUDA_SUCCESS &&
          mtype == CU_MEMORYTYPE_DEVICE && ordinal == dev && size > 0) {
        if (nr < kMaxRanges) {
          lo[nr] = static_cast<uintptr_t>(start);
          hi[nr] = static_cast<uintptr_t>(start) + size;
          ++nr;
        }
        continue;
      }
    }
    KAIO_TRY_FN(check_one_on_device(s[i], dev));
  }
  return KAIO_OK;
}

int zero_outputs(const Span* out, int n, cudaStream_t stream) {
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaMemsetAsync(const_cast<void*>(out[i].p), 0, out[i].bytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (K == 0)");
  }
  return KAIO_OK;
}

#define KAIO_TRY(expr)           \
  do {                           \
    const int st__ = (expr);     \
    if (st__ != KAIO_OK) return st__; \
  } while (0)

// The checks every projection entry makes after its own null-pointer and
// dimension rules, in this order: 16-byte alignment, size limits (packed
// words of one weight tensor, M x K), overlap, the current device, the empty
// problem (M == 0 or N == 0: nothing to do), output residency, K == 0 (the
// outputs are the empty sum: zeroed here), input residency. *run is set when
// the caller must launch a kernel; *dev and *info then describe the device.
int check_projection(const Span* in, int n_in, const Span* out, uint64_t packed_words, uint32_t M,
                     uint32_t N, uint32_t K, cudaStream_t stream, bool* run, int* dev, DeviceInfo* info) {
  *run = false;
  KAIO_TRY(check_aligned(in, n_in));
  KAIO_TRY(check_aligned(out, 3));
  if (packed_words > 0x7FFFFFFFull || static_cast<uint64_t>(M) * K > (1ull << 40))
    return fail(KAIO_ERR_INVALID_VALUE, "problem too large (M=%u N=%u K=%u)", M, N, K);
  KAIO_TRY(check_overlap(in, n_in, out, 3));
  KAIO_TRY(current_device(dev, info));
  if (M == 0 || N == 0) return KAIO_OK;
  KAIO_TRY(check_on_device(out, 3, *dev));
  if (K == 0) return zero_outputs(out, 3, stream);
  KAIO_TRY(check_on_device(in, n_in, *dev));
  *run = true;
  return KAIO_OK;
}

}  // namespace

namespace kaio {
// tc_decode.cu: the decode kernel's two-instruction routine alone (debug
// variant 2); declared here, its only caller.
cudaError_t launch_dequant_fast_debug(const uint32_t* w, const __half* s, __half* out, int K, int N,
                                      cudaStream_t stream);
}  // namespace kaio

extern "C" {

const char* kaio_last_error(void) { return g_last_error.c_str(); }

const char* kaio_status_string(int status) {
  switch (status) {
    case KAIO_OK: return "KAIO_OK";
    case KAIO_ERR_INVALID_VALUE: return "KAIO_ERR_INVALID_VALUE";
    case KAIO_ERR_MISALIGNED: return "KAIO_ERR_MISALIGNED";
    case KAIO_ERR_UNSUPPORTED_DEVICE: return "KAIO_ERR_UNSUPPORTED_DEVICE";
    case KAIO_ERR_CUDA: return "KAIO_ERR_CUDA";
    case KAIO_ERR_DEVICE_TIMEOUT: return "KAIO_ERR_DEVICE_TIMEOUT";
    default: return "unknown kaio_status";
  }
}

int kaio_qkv_path(uint32_t M) { return M <= 16 ? 0 : 1; }

int kaio_qkv_project_int4(const void* x, const uint32_t* wq, const uint32_t* wk, const uint32_t* wv,
                          const void* sq, const void* sk, const void* sv, void* q, void* k, void* v,
                          uint32_t M, uint32_t N, uint32_t K, kaio_stream_t stream_) {
  g_last_error.clear();
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t m = M, n = N, kk = K;
  const Span in[7] = {{"x", x, m * kk * 2},          {"w_q_packed", wq, kk / 8 * n * 4},
                      {"w_k_packed", wk, kk / 8 * n * 4}, {"w_v_packed", wv, kk / 8 * n * 4},
                      {"scales_q", sq, kk / 128 * n * 2}, {"scales_k", sk, kk / 128 * n * 2},
                      {"scales_v", sv, kk / 128 * n * 2}};
  const Span out[3] = {{"q", q, m * n * 2}, {"k", k, m * n * 2}, {"v", v, m * n * 2}};
  KAIO_TRY(check_not_null(in, 7));
  KAIO_TRY(check_not_null(out, 3));
  if (K % 128 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "K (%u) must be a multiple of group_size (128)", K);
  if (N % 8 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "N (%u) must be a multiple of 8 (16-byte rows)", N);
  bool run;
  int dev;
  DeviceInfo info;
  KAIO_TRY(check_projection(in, 7, out, static_cast<uint64_t>(K) / 8 * N, M, N, K, stream, &run, &dev, &info));
  if (!run) return KAIO_OK;

  const uint32_t* w3[3] = {wq, wk, wv};
  const __half* s3[3] = {static_cast<const __half*>(sq), static_cast<const __half*>(sk),
                         static_cast<const __half*>(sv)};
  __half* o3[3] = {static_cast<__half*>(q), static_cast<__half*>(k), static_cast<__half*>(v)};

  cudaError_t e;
  if (kaio_qkv_path(M) == 0) {
    const kaio::TcDecodePlan tp = kaio::plan_tc_decode(static_cast<int>(M), static_cast<int>(N),
                                                       static_cast<int>(K), dev);
    if (tp.ok) {
      e = kaio::launch_tc_decode(static_cast<const __half*>(x), w3, s3, o3, static_cast<int>(M),
                                 static_cast<int>(N), static_cast<int>(K), tp, stream);
      if (e != cudaSuccess) return cuda_fail(e, "tcgen05 decode kernel launch");
      return KAIO_OK;
    }
  }
  // M >= 17, or no cluster shape of the decode kernel can be resident: the
  // tile kernel (it takes any M; x rows past M are zero-filled by TMA).
  e = kaio::launch_tc_w4a16(static_cast<const __half*>(x), w3, s3, o3, static_cast<int>(M),
                            static_cast<int>(N), static_cast<int>(K), info.sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 W4A16 kernel launch");
  return KAIO_OK;
}

int kaio_debug_decode_wait_limit(const void* x, const uint32_t* wq, const uint32_t* wk, const uint32_t* wv,
                                 const void* sq, const void* sk, const void* sv, void* q, void* k, void* v,
                                 uint32_t M, uint32_t N, uint32_t K, uint64_t wait_limit_ns,
                                 kaio_stream_t stream_) {
  g_last_error.clear();
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t m = M, n = N, kk = K;
  const Span in[7] = {{"x", x, m * kk * 2},          {"w_q_packed", wq, kk / 8 * n * 4},
                      {"w_k_packed", wk, kk / 8 * n * 4}, {"w_v_packed", wv, kk / 8 * n * 4},
                      {"scales_q", sq, kk / 128 * n * 2}, {"scales_k", sk, kk / 128 * n * 2},
                      {"scales_v", sv, kk / 128 * n * 2}};
  const Span out[3] = {{"q", q, m * n * 2}, {"k", k, m * n * 2}, {"v", v, m * n * 2}};
  KAIO_TRY(check_not_null(in, 7));
  KAIO_TRY(check_not_null(out, 3));
  if (M == 0 || M > 16)
    return fail(KAIO_ERR_INVALID_VALUE, "M (%u) must be 1..16: this entry runs the decode kernel", M);
  if (K == 0 || K % 128 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "K (%u) must be a positive multiple of group_size (128)", K);
  if (N == 0 || N % 8 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "N (%u) must be a positive multiple of 8", N);
  bool run;
  int dev;
  DeviceInfo info;
  KAIO_TRY(check_projection(in, 7, out, static_cast<uint64_t>(K) / 8 * N, M, N, K, stream, &run, &dev, &info));
  if (!run) return KAIO_OK;
  const kaio::TcDecodePlan tp = kaio::plan_tc_decode(static_cast<int>(M), static_cast<int>(N),
                                                     static_cast<int>(K), dev);
  if (!tp.ok) return fail(KAIO_ERR_CUDA, "no resident launch shape for the decode kernel");
  const uint32_t* w3[3] = {wq, wk, wv};
  const __half* s3[3] = {static_cast<const __half*>(sq), static_cast<const __half*>(sk),
                         static_cast<const __half*>(sv)};
  __half* o3[3] = {static_cast<__half*>(q), static_cast<__half*>(k), static_cast<__half*>(v)};
  const cudaError_t e = kaio::launch_tc_decode_wait_limit(static_cast<const __half*>(x), w3, s3, o3,
                                                          static_cast<int>(M), static_cast<int>(N),
                                                          static_cast<int>(K), tp, wait_limit_ns, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 decode kernel launch");
  return KAIO_OK;
}

int kaio_qkv_project_int8(const void* x, const uint32_t* wq, const uint32_t* wk, const uint32_t* wv,
                          float scale_q, float scale_k, float scale_v, void* q, void* k, void* v,
                          uint32_t M, uint32_t N, uint32_t K, kaio_stream_t stream_) {
  g_last_error.clear();
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t m = M, n = N, kk = K;
  const Span in[4] = {{"x", x, m * kk * 2},
                      {"w_q_packed", wq, kk / 4 * n * 4},
                      {"w_k_packed", wk, kk / 4 * n * 4},
                      {"w_v_packed", wv, kk / 4 * n * 4}};
  const Span out[3] = {{"q", q, m * n * 2}, {"k", k, m * n * 2}, {"v", v, m * n * 2}};
  KAIO_TRY(check_not_null(in, 4));
  KAIO_TRY(check_not_null(out, 3));
  if (K % 128 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "K (%u) must be a multiple of 128 (the kernels' K group)", K);
  if (N % 8 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "N (%u) must be a multiple of 8 (16-byte rows)", N);
  bool run;
  int dev;
  DeviceInfo info;
  KAIO_TRY(check_projection(in, 4, out, static_cast<uint64_t>(K) / 4 * N, M, N, K, stream, &run, &dev, &info));
  if (!run) return KAIO_OK;

  const uint32_t* w3[3] = {wq, wk, wv};
  const float sc3[3] = {scale_q, scale_k, scale_v};
  __half* o3[3] = {static_cast<__half*>(q), static_cast<__half*>(k), static_cast<__half*>(v)};
  cudaError_t e;
  if (kaio_qkv_path(M) == 0) {
    const kaio::TcDecodePlan tp = kaio::plan_tc_decode_int8(static_cast<int>(M), static_cast<int>(N),
                                                            static_cast<int>(K), dev);
    if (tp.ok) {
      e = kaio::launch_tc_decode_int8(static_cast<const __half*>(x), w3, sc3, o3, static_cast<int>(M),
                                      static_cast<int>(N), static_cast<int>(K), tp, stream);
      if (e != cudaSuccess) return cuda_fail(e, "tcgen05 W8A16 decode kernel launch");
      return KAIO_OK;
    }
  }
  e = kaio::launch_tc_w8a16(static_cast<const __half*>(x), w3, sc3, o3, static_cast<int>(M),
                            static_cast<int>(N), static_cast<int>(K), info.sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 W8A16 kernel launch");
  return KAIO_OK;
}

int kaio_qkv_project_int4_noalloc(const void* x, const uint32_t* wq, const uint32_t* wk,
                                  const uint32_t* wv, const void* sq, const void* sk, const void* sv,
                                  void* q, void* k, void* v, uint32_t M, uint32_t N, uint32_t K,
                                  kaio_stream_t stream_) {
  g_last_error.clear();
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t m = M, n = N, kk = K;
  const Span in[7] = {{"x", x, m * kk * 2},          {"w_q_packed", wq, kk / 8 * n * 4},
                      {"w_k_packed", wk, kk / 8 * n * 4}, {"w_v_packed", wv, kk / 8 * n * 4},
                      {"scales_q", sq, kk / 128 * n * 2}, {"scales_k", sk, kk / 128 * n * 2},
                      {"scales_v", sv, kk / 128 * n * 2}};
  const Span out[3] = {{"q", q, m * n * 2}, {"k", k, m * n * 2}, {"v", v, m * n * 2}};
  KAIO_TRY(check_not_null(in, 7));
  KAIO_TRY(check_not_null(out, 3));
  if (M > 16)
    return fail(KAIO_ERR_INVALID_VALUE,
                "M (%u) exceeds 16: the allocation-free entry runs the decode kernel only", M);
  if (K % 128 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "K (%u) must be a multiple of group_size (128)", K);
  if (N % 8 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "N (%u) must be a multiple of 8 (16-byte rows)", N);
  const uint64_t groups = 3ull * ((static_cast<uint64_t>(N) + 255) / 256);
  if (groups > static_cast<uint64_t>(kaio::noalloc_max_counters()))
    return fail(KAIO_ERR_INVALID_VALUE,
                "N (%u) exceeds the allocation-free limit (%d column groups of 256 in its "
                "fixed %zu-byte scratch)", N, kaio::noalloc_max_counters(), kaio::kNoAllocScratchBytes);
  bool run;
  int dev;
  DeviceInfo info;
  KAIO_TRY(check_projection(in, 7, out, static_cast<uint64_t>(K) / 8 * N, M, N, K, stream, &run, &dev, &info));
  if (!run) return KAIO_OK;
  kaio::DecodeParams prm{};
  prm.x = static_cast<const __half*>(x);
  const uint32_t* w3[3] = {wq, wk, wv};
  const void* s3[3] = {sq, sk, sv};
  void* o3[3] = {q, k, v};
  for (int i = 0; i < 3; ++i) {
    prm.w[i] = w3[i];
    prm.s[i] = static_cast<const __half*>(s3[i]);
    prm.out[i] = static_cast<__half*>(o3[i]);
  }
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(N);
  prm.K = static_cast<int>(K);
  const cudaError_t e = kaio::launch_decode_noalloc(prm, dev, info.sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "allocation-free decode launch");
  return KAIO_OK;
}

namespace {

// C = A @ B with the result stored as f32 (esize 4) or f16 (esize 2).
int matmul_impl(const void* a, const void* b, void* c, size_t esize, uint32_t M, uint32_t N,
                uint32_t K, cudaStream_t stream) {
  const size_t m = M, n = N, kk = K;
  const Span in[2] = {{"a", a, m * kk * 2}, {"b", b, kk * n * 2}};
  const Span out[1] = {{"c", c, m * n * esize}};
  KAIO_TRY(check_not_null(in, 2));
  KAIO_TRY(check_not_null(out, 1));
  if (K % 8 != 0 || N % 8 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "K (%u) and N (%u) must be multiples of 8 (16-byte rows)", K, N);
  KAIO_TRY(check_aligned(in, 2));
  KAIO_TRY(check_aligned(out, 1));
  KAIO_TRY(check_overlap(in, 2, out, 1));
  int dev;
  DeviceInfo info;
  KAIO_TRY(current_device(&dev, &info));
  if (M == 0 || N == 0) return KAIO_OK;
  if (K == 0) {
    KAIO_TRY(check_on_device(out, 1, dev));
    return zero_outputs(out, 1, stream);
  }
  KAIO_TRY(check_on_device(in, 2, dev));
  KAIO_TRY(check_on_device(out, 1, dev));
  cudaError_t e = kaio::launch_tc_gemm(a, b, c, {static_cast<int>(M), static_cast<int>(N), static_cast<int>(K)},
                                       /*a_mn=*/false, /*b_mn=*/true, esize == 2, info.sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 matmul launch");
  return KAIO_OK;
}

// (dA, dB) = (G @ B^T, A^T @ G) stored as f32 (esize 4) or f16 (esize 2).
int matmul_backward_impl(const void* a, const void* b, const void* g, void* da, void* db,
                         size_t esize, uint32_t M, uint32_t N, uint32_t K, cudaStream_t stream) {
  const size_t m = M, n = N, kk = K;
  const Span in[3] = {{"a", a, m * kk * 2}, {"b", b, kk * n * 2}, {"g", g, m * n * 2}};
  const Span out[2] = {{"da", da, m * kk * esize}, {"db", db, kk * n * esize}};
  KAIO_TRY(check_not_null(in, 3));
  KAIO_TRY(check_not_null(out, 2));
  if (K % 8 != 0 || N % 8 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "K (%u) and N (%u) must be multiples of 8 (16-byte rows)", K, N);
  KAIO_TRY(check_aligned(in, 3));
  KAIO_TRY(check_aligned(out, 2));
  KAIO_TRY(check_overlap(in, 3, out, 2));
  int dev;
  DeviceInfo info;
  KAIO_TRY(current_device(&dev, &info));
  if (K == 0) return KAIO_OK;                      // dA [M,0] and dB [0,N] are empty
  if (M == 0 || N == 0) {
    // Empty contraction for the non-empty output: it is all zeros.
    KAIO_TRY(check_on_device(out, 2, dev));
    return zero_outputs(out, 2, stream);
  }
  KAIO_TRY(check_on_device(in, 3, dev));
  KAIO_TRY(check_on_device(out, 2, dev));
  const bool f16 = esize == 2;
  // dA[M, K] = G[M, N] @ B^T: Aop = G stored [M][N] (K-major over N);
  //   Bop = B^T, an N x K operand whose storage B[K][N] is [No][Ko] (K-major).
  cudaError_t e = kaio::launch_tc_gemm(g, b, da, {static_cast<int>(M), static_cast<int>(K), static_cast<int>(N)},
                                       false, false, f16, info.sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 matmul launch (dA)");
  // dB[K, N] = A^T @ G: Aop = A^T, a K x M operand stored A[M][K] = [Ko][Mo]
  //   (MN-major); Bop = G, M x N stored [Ko][No] (MN-major).
  e = kaio::launch_tc_gemm(a, g, db, {static_cast<int>(K), static_cast<int>(N), static_cast<int>(M)},
                           true, true, f16, info.sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 matmul launch (dB)");
  return KAIO_OK;
}

}  // namespace

int kaio_matmul_tc(const void* a, const void* b, float* c, uint32_t M, uint32_t N, uint32_t K,
                   kaio_stream_t stream) {
  g_last_error.clear();
  return matmul_impl(a, b, c, 4, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

int kaio_matmul_tc_f16(const void* a, const void* b, void* c, uint32_t M, uint32_t N, uint32_t K,
                       kaio_stream_t stream) {
  g_last_error.clear();
  return matmul_impl(a, b, c, 2, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

int kaio_matmul_tc_backward(const void* a, const void* b, const void* g, float* da, float* db,
                            uint32_t M, uint32_t N, uint32_t K, kaio_stream_t stream) {
  g_last_error.clear();
  return matmul_backward_impl(a, b, g, da, db, 4, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

int kaio_matmul_tc_backward_f16(const void* a, const void* b, const void* g, void* da, void* db,
                                uint32_t M, uint32_t N, uint32_t K, kaio_stream_t stream) {
  g_last_error.clear();
  return matmul_backward_impl(a, b, g, da, db, 2, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

bool float_type(int dtype, kaio::FloatType* t, size_t* esize) {
  switch (dtype) {
    case KAIO_DTYPE_F32: *t = kaio::FloatType::F32; *esize = 4; return true;
    case KAIO_DTYPE_F64: *t = kaio::FloatType::F64; *esize = 8; return true;
    case KAIO_DTYPE_F16: *t = kaio::FloatType::F16; *esize = 2; return true;
    case KAIO_DTYPE_BF16: *t = kaio::FloatType::BF16; *esize = 2; return true;
    default: return false;
  }
}

// Shared by the per-group dequantisation and its backward, in the order the
// page's plan checks them: element types, sizes and group, empty problem (Ok,
// no launch), then pointers (null, alignment to the element size, overlap,
// residency) and the device.
int dequant_group_impl(bool backward, int dtype, int q_dtype, int32_t outer, int32_t axis, int32_t group,
                       const void* in, const void* scale, void* out, cudaStream_t stream) {
  kaio::FloatType t;
  size_t es;
  if (!float_type(dtype, &t, &es))
    return fail(KAIO_ERR_INVALID_VALUE, "unsupported float type %d (f32, f64, f16 or bf16)", dtype);
  if (q_dtype != KAIO_DTYPE_S8 && q_dtype != KAIO_DTYPE_U8)
    return fail(KAIO_ERR_INVALID_VALUE, "the quantised type must be S8 or U8 (got %d)", q_dtype);
  if (outer < 0 || axis < 0)
    return fail(KAIO_ERR_INVALID_VALUE, "outer (%d) and axis (%d) must be non-negative", outer, axis);
  if (group <= 0) return fail(KAIO_ERR_INVALID_VALUE, "group (%d) must be > 0", group);
  if (axis % group != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "axis (%d) must be a multiple of group (%d)", axis, group);
  const size_t total = static_cast<size_t>(outer) * static_cast<size_t>(axis);
  if (total == 0) return KAIO_OK;
  const size_t in_es = backward ? es : 1;
  const char* in_name = backward ? "dy" : "q";
  const char* out_name = backward ? "dx" : "out";
  const Span sin{in_name, in, total * in_es};
  const Span ssc{"scale", scale, static_cast<size_t>(outer) * (static_cast<size_t>(axis) / group) * es};
  const Span sout{out_name, out, total * es};
  const Span all[3] = {sin, ssc, sout};
  KAIO_TRY(check_not_null(all, 3));
  const size_t align[3] = {in_es, es, es};
  for (int i = 0; i < 3; ++i)
    if (reinterpret_cast<uintptr_t>(all[i].p) % align[i] != 0)
      return fail(KAIO_ERR_MISALIGNED, "%s (%p) is not aligned to its %zu-byte elements", all[i].name,
                  all[i].p, align[i]);
  if (overlaps(sout, ssc)) return fail(KAIO_ERR_INVALID_VALUE, "%s overlaps scale", out_name);
  // The backward may run in place (dx == dy); any other overlap is an error.
  if (overlaps(sout, sin) && !(backward && in == out))
    return fail(KAIO_ERR_INVALID_VALUE, "%s overlaps %s (only dx == dy exactly is allowed)", out_name, in_name);
  int dev;
  DeviceInfo info;
  KAIO_TRY(current_device(&dev, &info));
  KAIO_TRY(check_on_device(all, 3, dev));
  const cudaError_t e =
      backward ? kaio::launch_dequant_group_backward(t, in, scale, out, outer, axis, group, info.sms, stream)
               : kaio::launch_dequant_group_forward(t, q_dtype == KAIO_DTYPE_U8, in, scale, out, outer, axis,
                                                    group, info.sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "per-group dequantisation launch");
  return KAIO_OK;
}

}  // namespace

int kaio_dequantize_per_group_backward(int dtype, int q_dtype, int32_t outer, int32_t axis, int32_t group,
                                       const void* dy, const void* scale, void* dx, kaio_stream_t stream) {
  g_last_error.clear();
  return dequant_group_impl(true, dtype, q_dtype, outer, axis, group, dy, scale, dx,
                            reinterpret_cast<cudaStream_t>(stream));
}

int kaio_dequantize_per_group(int q_dtype, int dtype, int32_t outer, int32_t axis, int32_t group,
                              const void* q, const void* scale, void* out, kaio_stream_t stream) {
  g_last_error.clear();
  return dequant_group_impl(false, dtype, q_dtype, outer, axis, group, q, scale, out,
                            reinterpret_cast<cudaStream_t>(stream));
}

int kaio_dequant_int4_debug(const uint32_t* w, const void* s, void* out, uint32_t K, uint32_t N,
                            int variant, kaio_stream_t stream_) {
  g_last_error.clear();
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t n = N, kk = K;
  const Span in[2] = {{"w", w, kk / 8 * n * 4}, {"s", s, kk / 128 * n * 2}};
  const Span o[1] = {{"out", out, kk * n * 2}};
  KAIO_TRY(check_not_null(in, 2));
  KAIO_TRY(check_not_null(o, 1));
  if (K % 128 != 0)
    return fail(KAIO_ERR_INVALID_VALUE, "K (%u) must be a multiple of group_size (128)", K);
  if (N % 8 != 0) return fail(KAIO_ERR_INVALID_VALUE, "N (%u) must be a multiple of 8", N);
  if (variant < 0 || variant > 2)
    return fail(KAIO_ERR_INVALID_VALUE, "variant (%d) must be 0, 1 or 2", variant);
  KAIO_TRY(check_aligned(in, 2));
  KAIO_TRY(check_aligned(o, 1));
  KAIO_TRY(check_overlap(in, 2, o, 1));
  int dev;
  DeviceInfo info;
  KAIO_TRY(current_device(&dev, &info));
  if (K == 0 || N == 0) return KAIO_OK;
  KAIO_TRY(check_on_device(in, 2, dev));
  KAIO_TRY(check_on_device(o, 1, dev));
  cudaError_t e =
      variant == 2 ? kaio::launch_dequant_fast_debug(w, static_cast<const __half*>(s), static_cast<__half*>(out),
                                                     static_cast<int>(K), static_cast<int>(N), stream)
                   : kaio::launch_dequant_debug(w, static_cast<const __half*>(s), static_cast<__half*>(out),
                                                static_cast<int>(K), static_cast<int>(N), variant, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dequant kernel launch");
  return KAIO_OK;
}

int kaio_device_status(void) {
  g_last_error.clear();
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  const unsigned err_tc = kaio::read_and_clear_tc_errors();
  const unsigned err_td = kaio::read_and_clear_tc_decode_errors();
  if (err_tc == 0xFFFFFFFFu || err_td == 0xFFFFFFFFu)
    return fail(KAIO_ERR_CUDA, "could not read the device error word");
  const unsigned err = err_tc | err_td;
  if (err & kaio::kDevErrTimeoutHost)
    return fail(KAIO_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (device error word 0x%x)", err);
  return KAIO_OK;
}

}  // extern "C"
