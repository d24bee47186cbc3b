// Internal to libpkv: the model geometry and the device helpers that the
// decode (pkv.cu) and prefill (prefill.cu) kernels share: shared-memory
// addresses, the sticky error word, mbarriers with bounded waits, the base-2
// exponential and BF16 packing.
//
// Geometry [6 Hours of YouTube and 85 handtyped pages of notes on LLM
// Inference - Start here, README feature list: 32 query heads over 8 KV heads,
// head_dim 64, 16-token pages, 2048-token context].
#ifndef PKV_DEVICE_COMMON_CUH
#define PKV_DEVICE_COMMON_CUH

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv_dev {

constexpr int kPage = 16;                       // tokens per page
constexpr int kHq = 32;                         // query heads
constexpr int kHkv = 8;                         // KV heads
constexpr int kGroup = kHq / kHkv;              // query heads per KV head
constexpr int kDim = 64;                        // head_dim
constexpr int kMaxSeqLen = 2048;
constexpr int kMaxPages = kMaxSeqLen / kPage;   // block-table row length
constexpr int kRowBytes = kDim * 2;             // one token of one kv head: 128 B

// about two seconds at the maximum SM clock
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_error(int* err, int bits) { atomicOr(err, bits); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One try_wait on an mbarrier phase, without a suspend-time hint (the
// instruction returns after the hardware's own time limit): measured on
// GB300, the hand-offs between warps come out shorter than with a long hint
// (prefill attention +1.1 %, decode +0.2 to +1.1 %).
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait on an mbarrier phase: false after about two seconds.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > kWaitCycles) return false;
  }
  return true;
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// 2^x by the SFU's approximate exponential (PTX ex2.approx.ftz.f32: relative
// error about 2^-22; results below 2^-126, i.e. softmax weights that cannot
// contribute, flush to zero; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two FP32 values -> BF16 pair (element 0 in the low half), each rounded to
// nearest, ties to even.
__device__ __forceinline__ uint32_t float2_to_bf16x2(float e0, float e1) {
  uint32_t w;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(e1), "f"(e0));
  return w;
}

}  // namespace pkv_dev

#endif  // PKV_DEVICE_COMMON_CUH
