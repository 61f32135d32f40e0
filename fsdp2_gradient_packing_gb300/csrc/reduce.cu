// The emulated reduce-scatter (fsdp_emulated_reduce_scatter), a one-GPU
// stand-in for the collective that tests and benchmarks put between the pack
// and the reduce-scatter copy-out, and the plain streaming widen
// (fsdp_debug_stream_widen) that benchmarks time beside the pack.  Neither is
// a step of the packing path; they share the host-side argument checks and
// the bit conversions of the table walker (kernels.cu, bf16_bits.h).
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "bf16_bits.h"
#include "layout.h"

namespace fsdp {
namespace {
// ---------------------------------------------------------------------------
// Emulated reduce-scatter (a test utility): out[i] = in_0[i] + in_1[i] + ...
// added over the inputs in order, each partial sum rounded to the element
// type -- FP32: one correctly rounded binary32 addition (no flush of
// subnormals); BF16: a binary32 addition of the two values, then round to
// nearest even to BF16; a NaN sum is the canonical quiet NaN.  The first
// input enters unchanged.  Every input and the output have the same shape.
// ---------------------------------------------------------------------------
constexpr int kMaxSumInputs = 256;
constexpr int kSumThreads = 256;

struct SumArgs {
  const void *in[kMaxSumInputs];
  void *out;
  int64_t n;      // elements
  int32_t n_in;
  int32_t head;   // leading elements before the first 16-byte boundary; -1: no vector path
};

// A NaN sum (a NaN operand, or infinities of opposite sign) becomes the
// canonical quiet NaN, so the result does not depend on the machine.
template <bool BF16>
__device__ __forceinline__ uint32_t add_bits(uint32_t acc, uint32_t x) {
  if constexpr (BF16) {
    const float s = __fadd_rn(__uint_as_float(acc << 16), __uint_as_float(x << 16));
    return (s != s) ? 0x7FC0u : f32_to_bf16_bits(__float_as_uint(s));
  } else {
    const float s = __fadd_rn(__uint_as_float(acc), __uint_as_float(x));
    return (s != s) ? 0x7FC00000u : __float_as_uint(s);
  }
}

// Two BF16 sums at once with the hardware's BF16 pair addition, which rounds
// each exact sum to nearest, ties to even.  That is the same result as
// add_bits<true>: adding two BF16 values in binary32 and rounding the sum to
// BF16 rounds twice, but binary32 keeps at least 2 x 8 + 1 significant bits,
// and with that margin a second rounding of a sum always lands where one
// rounding of the exact sum does.  NaN sums keep the hardware's payload here;
// canonical_nan_pair makes them the canonical quiet NaN.
__device__ __forceinline__ uint32_t add_bf16_raw(uint32_t x, uint32_t y) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(y));
  return d;
}

__device__ __forceinline__ uint32_t canonical_nan_pair(uint32_t d) {
  if ((d & 0x7FFFu) > 0x7F80u) d = (d & 0xFFFF0000u) | 0x7FC0u;
  if ((d & 0x7FFF0000u) > 0x7F800000u) d = (d & 0x0000FFFFu) | 0x7FC00000u;
  return d;
}

// Bit 15 or 31 set where that half of d is a NaN: a half h (sign dropped)
// is a NaN when h > 0x7F80, i.e. when h + 0x7F carries into bit 15.  The
// sum stays below 0x10000, so nothing carries into the other half.
__device__ __forceinline__ uint32_t nan_halves(uint32_t d) {
  return ((d & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u;
}

// Lane-wise sum of two 16-byte vectors of elements.  For BF16 the NaN
// fix-up runs only when one of the eight sums is a NaN.
template <bool BF16>
__device__ __forceinline__ uint4 add_vec(uint4 a, uint4 b) {
  if constexpr (BF16) {
    uint4 d = make_uint4(add_bf16_raw(a.x, b.x), add_bf16_raw(a.y, b.y), add_bf16_raw(a.z, b.z),
                         add_bf16_raw(a.w, b.w));
    if (nan_halves(d.x) | nan_halves(d.y) | nan_halves(d.z) | nan_halves(d.w))
      d = make_uint4(canonical_nan_pair(d.x), canonical_nan_pair(d.y), canonical_nan_pair(d.z),
                     canonical_nan_pair(d.w));
    return d;
  } else {
    return make_uint4(add_bits<false>(a.x, b.x), add_bits<false>(a.y, b.y), add_bits<false>(a.z, b.z),
                      add_bits<false>(a.w, b.w));
  }
}

template <bool BF16>
__device__ __forceinline__ void sum_scalar(const SumArgs &a, int64_t i) {
  if constexpr (BF16) {
    uint32_t acc = reinterpret_cast<const uint16_t *>(a.in[0])[i];
    for (int q = 1; q < a.n_in; ++q) acc = add_bits<true>(acc, reinterpret_cast<const uint16_t *>(a.in[q])[i]);
    reinterpret_cast<uint16_t *>(a.out)[i] = (uint16_t)acc;
  } else {
    uint32_t acc = reinterpret_cast<const uint32_t *>(a.in[0])[i];
    for (int q = 1; q < a.n_in; ++q) acc = add_bits<false>(acc, reinterpret_cast<const uint32_t *>(a.in[q])[i]);
    reinterpret_cast<uint32_t *>(a.out)[i] = acc;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kSumThreads) sum_kernel(const __grid_constant__ SumArgs a) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (a.head < 0) {
    for (int64_t i = tid; i < a.n; i += stride) sum_scalar<BF16>(a, i);
    return;
  }
  constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  const int64_t head = a.head < a.n ? a.head : a.n;
  const int64_t nvec = (a.n - head) / EPV;
  const int64_t tail0 = head + nvec * EPV;
  if (tid < head) sum_scalar<BF16>(a, tid);
  if (tail0 + tid < a.n) sum_scalar<BF16>(a, tail0 + tid);
  const int es = BF16 ? 2 : 4;
  // Two vectors per thread and round (v0 and v0 + stride), each summed over
  // the inputs in rank order, with up to eight 16-byte loads in flight.
  auto load = [&](int q, int64_t byte) {
    return __ldcs(reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(a.in[q]) + byte));
  };
  for (int64_t v0 = tid; v0 < nvec; v0 += 2 * stride) {
    const bool two = v0 + stride < nvec;
    const int64_t b0 = (head + v0 * EPV) * es, b1 = (head + (two ? v0 + stride : v0) * EPV) * es;
    uint4 acc0 = load(0, b0), acc1 = load(0, b1);
    for (int q = 1; q < a.n_in; q += 4) {
      uint4 x[4], y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (q + k < a.n_in) {
          x[k] = load(q + k, b0);
          y[k] = load(q + k, b1);
        }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (q + k < a.n_in) {
          acc0 = add_vec<BF16>(acc0, x[k]);
          acc1 = add_vec<BF16>(acc1, y[k]);
        }
    }
    *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(a.out) + b0) = acc0;
    if (two) *reinterpret_cast<uint4 *>(reinterpret_cast<char *>(a.out) + b1) = acc1;
  }
}

// ---------------------------------------------------------------------------
// Plain streaming widen (a measurement utility): dst[i] = bits(src[i]) << 16,
// BF16 to FP32, the pack's own 1 : 2 mix of bytes read to bytes written.
// Grid-stride over 16-byte vectors of the source; each thread loads one
// vector (streaming, read once) and stores the two 16-byte vectors it
// widens to, so every warp store covers 1 KiB of contiguous destination.
// ---------------------------------------------------------------------------
constexpr int kWidenThreads = 256;
constexpr int kWidenBlocksPerSm = 32;

__global__ void __launch_bounds__(kWidenThreads) widen_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                              int64_t nvec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const uint4 x = __ldcs(src + v);
    dst[2 * v] = make_uint4(x.x << 16, x.x & 0xFFFF0000u, x.y << 16, x.y & 0xFFFF0000u);
    dst[2 * v + 1] = make_uint4(x.z << 16, x.z & 0xFFFF0000u, x.w << 16, x.w & 0xFFFF0000u);
  }
}

}  // namespace
}  // namespace fsdp

using namespace fsdp;

extern "C" {

fsdp_status_t fsdp_emulated_reduce_scatter(const fsdp_layout_t *L, const void *const *packed,
                                           void *const *reduced, fsdp_stream_t stream) {
  fsdp_status_t st = check_layout(L);
  if (st != FSDP_OK) return st;
  const int B = (int)L->bucket.size(), W = L->W;
  if (W > kMaxSumInputs) return fail(FSDP_EUNSUPPORTED, "emulated reduce-scatter supports W <= 256");
  if (B > 0 && (!packed || !reduced)) return fail(FSDP_EINVAL, "packed or reduced is NULL");
  for (int b = 0; b < B; ++b) {
    const int64_t sz = dtype_bytes(L->bucket[b].dtype), bytes = (int64_t)W * L->bucket[b].S * sz;
    for (int q = 0; q < W; ++q)
      if ((st = check_ptr(packed[(int64_t)b * W + q], bytes, sz, "packed", (int64_t)b * W + q)) != FSDP_OK) return st;
    if ((st = check_ptr(reduced[b], bytes, sz, "reduced", b)) != FSDP_OK) return st;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int b = 0; b < B; ++b) {
    const int64_t n = (int64_t)W * L->bucket[b].S;
    if (n == 0) continue;
    const int sz = (int)dtype_bytes(L->bucket[b].dtype);
    SumArgs a;
    a.out = reduced[b];
    a.n = n;
    a.n_in = W;
    // The vector path needs every pointer at the same phase modulo 16 bytes.
    const uintptr_t phase = (uintptr_t)reduced[b] & 15u;
    bool same = true;
    for (int q = 0; q < W; ++q) {
      a.in[q] = packed[(int64_t)b * W + q];
      same = same && (((uintptr_t)a.in[q] & 15u) == phase);
    }
    a.head = same ? (int32_t)(((16u - phase) & 15u) / (unsigned)sz) : -1;
    const int64_t work = same ? n / (16 / sz) + 1 : n;
    int64_t grid = (work + kSumThreads - 1) / kSumThreads;
    const int64_t cap = (int64_t)(L->sms > 0 ? L->sms : 1) * 8;
    if (grid > cap) grid = cap;
    void *args[] = {&a};
    const void *fn = sz == 2 ? reinterpret_cast<const void *>(&sum_kernel<true>)
                             : reinterpret_cast<const void *>(&sum_kernel<false>);
    cudaError_t e = cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(kSumThreads), args, 0, s);
    if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("kernel launch failed: ") + cudaGetErrorString(e));
  }
  clear_error();
  return FSDP_OK;
}

fsdp_status_t fsdp_debug_stream_widen(const void *src, int64_t n, void *dst, fsdp_stream_t stream) {
  if (n < 0 || n % 8 != 0) return fail(FSDP_EINVAL, "n must be a non-negative multiple of 8");
  if (n == 0) {
    clear_error();
    return FSDP_OK;
  }
  if (!src || !dst) return fail(FSDP_EINVAL, "src or dst is NULL");
  if (((uintptr_t)src | (uintptr_t)dst) & 15u) return fail(FSDP_EINVAL, "src and dst must be 16-byte aligned");
  const uintptr_t s0 = (uintptr_t)src, s1 = s0 + (uintptr_t)n * 2, d0 = (uintptr_t)dst, d1 = d0 + (uintptr_t)n * 4;
  if (s0 < d1 && d0 < s1) return fail(FSDP_EINVAL, "src and dst overlap");
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("device query failed: ") + cudaGetErrorString(e));
  const int64_t nvec = n / 8;
  int64_t grid = (int64_t)(sms > 0 ? sms : 1) * kWidenBlocksPerSm;
  const int64_t need = (nvec + kWidenThreads - 1) / kWidenThreads;
  if (grid > need) grid = need;
  const uint4 *s = static_cast<const uint4 *>(src);
  uint4 *d = static_cast<uint4 *>(dst);
  void *args[] = {&s, &d, const_cast<int64_t *>(&nvec)};
  e = cudaLaunchKernel(reinterpret_cast<const void *>(&widen_kernel), dim3((unsigned)grid), dim3(kWidenThreads), args, 0,
                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FSDP_ECUDA, std::string("kernel launch failed: ") + cudaGetErrorString(e));
  clear_error();
  return FSDP_OK;
}

}  // extern "C"
