// Unit-rate microbenchmarks behind the MUFU-vs-tensor argument of "LLM
// Systems 22: Flash Attention", sections 4.1.2 and 4.2: per SM and per clock,
// how many exponentials the special-function unit retires (ex2.approx) and how
// many bf16 FLOPs tcgen05.mma retires.  Each kernel times itself with the SM
// cycle counter, so the results are in units per SM-clock whatever the clock.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "fa_kernels.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kChains = 8;  // independent dependency chains per thread
constexpr int kMaxSms = 1024;

// Per-CTA cycle counts (one CTA per SM) and a sink that keeps the timed loops
// from being optimised away.
__device__ unsigned long long g_cycles[kMaxSms];
__device__ float g_sink[kMaxSms];

// kind 0: ex2.approx.ftz.f32; 1: cvt.rn.bf16x2.f32; 2: fma.rn.f32.  The
// softmax's per-pair step, counted in exponentials: 3: two ex2 and one
// cvt.rn.bf16x2.f32; 5: the forward softmax's full step (paired FMA, two
// ex2, paired add into a row sum, cvt pack); 7: kind 5 with a quarter of the
// pairs through the polynomial exp2 (ex2_poly2) instead of the
// special-function unit.
template <int KIND>
__global__ void __launch_bounds__(1024, 1) unit_rate_kernel(int iters, unsigned long long* cycles, float* sink) {
  float x[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) x[c] = -1.0f - 0.001f * (threadIdx.x + c);
  uint64_t acc2[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) acc2[c] = f2_pack(0.f, 0.f);
  const uint64_t c2 = f2_pack(0.9f, 0.9f), n2 = f2_pack(-0.1f, -0.2f);
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      if constexpr (KIND == 0) {
        x[c] = ex2_approx(x[c]) - 1.5f;  // stays in (-1.5, -0.5): no denormals or overflow
      } else if constexpr (KIND == 1) {
        const uint32_t p = pack_bf16x2(x[c], x[c] + 1.0f);
        x[c] = __uint_as_float(p & 0xFFFF0000u) * 0.5f - 0.75f;
      } else if constexpr (KIND >= 3) {
        float x0 = x[c], x1 = x[c] - 0.25f;
        if constexpr (KIND >= 5) f2_unpack(ffma2(f2_pack(x0, x1), c2, n2), x0, x1);
        float a, b;
        if (KIND == 7 && (c & 3) == 3) {
          f2_unpack(ex2_poly2(x0, x1), a, b);
        } else {
          a = ex2_approx(x0);
          b = ex2_approx(x1);
        }
        if constexpr (KIND >= 5) acc2[c] = fadd2(acc2[c], f2_pack(a, b));
        const uint32_t pk = pack_bf16x2(a, b);
        x[c] = __uint_as_float(pk & 0xFFFF0000u) * -0.5f - 0.75f;  // stays in (-1.2, -0.8)
      } else {
        x[c] = fmaf(x[c], 0.999f, -0.001f);
      }
    }
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) {
    float a0, a1;
    f2_unpack(acc2[c], a0, a1);
    s += x[c] + a0 + a1;
  }
  if (s == 12345.f) sink[threadIdx.x % kMaxSms] = s;  // keeps the loop alive
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}
// Pseudo-random bf16 pair with magnitudes in [0.5, 1) and random signs.
__device__ __forceinline__ uint32_t random_bf16x2(uint32_t i) {
  uint32_t h = i * 0x9E3779B9u;
  h ^= h >> 15;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  const uint32_t lo = (h & 0x8000u) | 0x3F00u | (h & 0x7Fu);
  const uint32_t hi = ((h >> 16) & 0x8000u) | 0x3F00u | ((h >> 16) & 0x7Fu);
  return lo | (hi << 16);
}
// Accuracy of ex2_poly2 against ex2.approx.ftz.f32 over x in [-30, 8]
// (2^20 points): the largest relative difference, as fp32 bits in *out (a
// positive float orders as its bits).  Inputs far below the clamp (-1e4,
// -inf) must give a value in [0, 2^-100]; otherwise *bad is set.
__global__ void ex2_poly_accuracy_kernel(unsigned int* out, unsigned int* bad) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const float x0 = -30.0f + 38.0f * (static_cast<float>(i) / 1048576.0f);
  const float x1 = -30.0f + 38.0f * (static_cast<float>(i) + 0.5f) / 1048576.0f;
  float p0, p1;
  f2_unpack(ex2_poly2(x0, x1), p0, p1);
  const float e0 = fabsf(p0 / ex2_approx(x0) - 1.0f), e1 = fabsf(p1 / ex2_approx(x1) - 1.0f);
  atomicMax(out, __float_as_uint(fmaxf(e0, e1)));
  if (i == 0) {
    float q0, q1;
    f2_unpack(ex2_poly2(-1.0e4f, -CUDART_INF_F), q0, q1);
    if (!(q0 >= 0.0f && q0 <= 7.9e-31f && q1 >= 0.0f && q1 <= 7.9e-31f)) atomicOr(bad, 1u);
  }
}
// tcgen05.mma throughput: one thread issues `iters` x 4 MMAs of M=128, N, K=16
// (bf16, fp32 accumulate in TMEM; A from shared memory, or from TMEM when
// TS) and waits for them to finish.  Operands are zero, or pseudo-random bf16
// when RND (the realistic case: switching data draws more power than zeros).
template <int N, bool TS, bool RND>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters, unsigned long long* cycles, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gen = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  for (int i = threadIdx.x; i < (128 + N) * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gen)[i] =
        RND ? make_uint4(random_bf16x2(4 * i), random_bf16x2(4 * i + 1), random_bf16x2(4 * i + 2),
                         random_bf16x2(4 * i + 3))
            : make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done_bar), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (TS) {  // fill the A operand's 32 TMEM columns (128..159), each warp its lane quarter
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = RND ? random_bf16x2(threadIdx.x * 32 + i + 977u) : 0u;
    tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 128, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = idesc_bf16(128, N, false, false);
    const uint32_t sA = base, sB = base + 128 * 128;
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        if (TS)
          mma_ts(tmem, tmem + 128 + kk * 8, sdesc_sw128(sB + kk * 32, 16, 1024), idesc, (i | kk) ? 1u : 0u);
        else
          mma_ss(tmem, sdesc_sw128(sA + kk * 32, 16, 1024), sdesc_sw128(sB + kk * 32, 16, 1024), idesc,
                 (i | kk) ? 1u : 0u);
    }
    tc_commit(smem_u32(&done_bar));
    wait_drain(smem_u32(&done_bar), 0, err, 2000000000ull);
    const unsigned long long t1 = clock64();
    cycles[blockIdx.x] = t1 - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int N, bool TS, bool RND>
cudaError_t launch_mma_rate(int sms, int iters, unsigned long long* cyc, uint32_t* err, cudaStream_t s) {
  const int smem = (128 + N) * 128 + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(mma_rate_kernel<N, TS, RND>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_rate_kernel<N, TS, RND><<<sms, 128, smem, s>>>(iters, cyc, err);
  return cudaGetLastError();
}
// The forward kernel's MMA stream without its softmax: per iteration and per
// query tile t, O_t += P_t V (A from TMEM, 8 x K16) then S_t = Q K^T (both
// from shared memory, 8 x K16), pseudo-random bf16 operands.  TMEM: S_t at
// columns 128t; with ALIAS the P_t operand lies in S_t's first 64 columns
// (so each S_t overwrites what the preceding PV_t read), otherwise in
// columns 384 + 64t that no MMA writes.  SPLIT issues both PVs before both
// S's.  The rate says how fast the tensor pipe retires this stream when no
// other unit holds it up (the forward kernel's aliasing of P over S and its
// MMA order cost the pipe nothing if it is the rate of separate operands).
// The operand descriptors are formed as in the forward kernel (tile bases
// once, a 64-bit add per K step).
template <int DPV, bool ALIAS, bool SPLIT>
__global__ void __launch_bounds__(128, 1) fwd_stream_kernel(int iters, unsigned long long* cycles, uint32_t* err) {
  static_assert(ALIAS || DPV == 64, "separate P columns fit only beside 64-column O tiles");
  constexpr int TILE = 128 * 128 * 2;  // one 128 x 128 bf16 tile: two 128-byte swizzled 64-column blocks
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gen = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  for (int i = threadIdx.x; i < 3 * TILE / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gen)[i] =
        make_uint4(random_bf16x2(4 * i), random_bf16x2(4 * i + 1), random_bf16x2(4 * i + 2), random_bf16x2(4 * i + 3));
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done_bar), 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (warp < 4) {  // pseudo-random bf16 in every column an MMA may read as P before it is written
    uint32_t z[32];
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c = 0; c < 512; c += 32) {
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = random_bf16x2(threadIdx.x * 512 + c + i + 977u);
      tmem_st32(lane_base + c, z);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(128, DPV, false, true);
    const uint32_t sQ = base, sK = base + TILE, sV = base + 2 * TILE;
    auto s_col = [](int t) -> uint32_t { return 128u * t; };
    auto o_col = [](int t) -> uint32_t { return 256u + DPV * t; };
    auto p_col = [](int t) -> uint32_t { return ALIAS ? 128u * t : 384u + 64u * t; };
    const uint64_t dV = sdesc_sw128(sV, 128 * 128, 1024), dQ = sdesc_sw128(sQ, 16, 1024), dK = sdesc_sw128(sK, 16, 1024);
    uint64_t dVi = dV, dKi = dK;  // this iteration's V and K operands
    auto pv = [&](int t) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tmem + o_col(t), tmem + p_col(t) + kk * 8, sdesc_add(dVi, kk * 2048), idesc_o, 1u);
    };
    auto sg = [&](int t) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (kk / 4) * (128 * 128) + (kk % 4) * 32;
        mma_ss(tmem + s_col(t), sdesc_add(dQ, koff), sdesc_add(dKi, koff), idesc_s, kk > 0 ? 1u : 0u);
      }
    };
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      if (SPLIT) {
        pv(0); pv(1); sg(0); sg(1);
      } else {
        pv(0); sg(0); pv(1); sg(1);
      }
    }
    tc_commit(smem_u32(&done_bar));
    wait_drain(smem_u32(&done_bar), 0, err, 2000000000ull);
    const unsigned long long t1 = clock64();
    cycles[blockIdx.x] = t1 - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DPV, bool ALIAS, bool SPLIT>
cudaError_t launch_fwd_stream(int sms, int iters, unsigned long long* cyc, uint32_t* err, cudaStream_t s) {
  const int smem = 3 * 128 * 128 * 2 + 1024;
  auto kern = fwd_stream_kernel<DPV, ALIAS, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<sms, 128, smem, s>>>(iters, cyc, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t run_microbench(int which, int iters, uint32_t* err, double* result, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (sms > kMaxSms) sms = kMaxSms;
  unsigned long long* cyc = nullptr;
  float* sink = nullptr;
  if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&cyc), g_cycles)) != cudaSuccess) return e;
  if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&sink), g_sink)) != cudaSuccess) return e;
  double units_per_cta = 0;
  const int threads = 1024;
  switch (which) {
    case 0: unit_rate_kernel<0><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 1: unit_rate_kernel<1><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 2: unit_rate_kernel<2><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 38: unit_rate_kernel<3><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 40: unit_rate_kernel<5><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 43: unit_rate_kernel<7><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 42: {  // accuracy, not a rate
      unsigned int* acc = reinterpret_cast<unsigned int*>(cyc);
      if ((e = cudaMemsetAsync(acc, 0, 2 * sizeof(unsigned int), s)) != cudaSuccess) return e;
      ex2_poly_accuracy_kernel<<<4096, 256, 0, s>>>(acc, acc + 1);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      unsigned int h[2];
      if ((e = cudaMemcpyAsync(h, acc, sizeof(h), cudaMemcpyDeviceToHost, s)) != cudaSuccess) return e;
      if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
      float r;
      memcpy(&r, &h[0], sizeof(r));
      *result = h[1] ? -1.0 : static_cast<double>(r);
      return cudaSuccess;
    }
    case 3: e = launch_mma_rate<256, false, false>(sms, iters, cyc, err, s); break;
    case 4: e = launch_mma_rate<128, false, false>(sms, iters, cyc, err, s); break;
    case 5: e = launch_mma_rate<128, true, false>(sms, iters, cyc, err, s); break;
    case 6: e = launch_mma_rate<256, false, true>(sms, iters, cyc, err, s); break;
    case 7: e = launch_mma_rate<128, true, true>(sms, iters, cyc, err, s); break;
    case 8: e = launch_fwd_stream<128, true, false>(sms, iters, cyc, err, s); break;
    case 9: e = launch_fwd_stream<64, true, false>(sms, iters, cyc, err, s); break;
    case 10: e = launch_fwd_stream<64, false, false>(sms, iters, cyc, err, s); break;
    case 11: e = launch_fwd_stream<128, true, true>(sms, iters, cyc, err, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if (which <= 2)
    units_per_cta = static_cast<double>(threads) * iters * kChains;
  else if (which >= 38)  // two exponentials per step (38, 40, 43)
    units_per_cta = 2.0 * threads * iters * kChains;
  else if (which <= 7)
    units_per_cta = 2.0 * 128 * ((which == 3 || which == 6) ? 256 : 128) * 64 * static_cast<double>(iters);
  else  // two query tiles x (S: 128 x 128 x 128, PV: 128 x DPV x 128)
    units_per_cta = 2.0 * (2.0 * 128 * 128 * 128 + 2.0 * 128 * ((which == 9 || which == 10) ? 64 : 128) * 128) *
                    static_cast<double>(iters);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  static unsigned long long host_cyc[kMaxSms];
  if ((e = cudaMemcpy(host_cyc, cyc, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return e;
  double acc = 0;
  for (int i = 0; i < sms; ++i) acc += units_per_cta / static_cast<double>(host_cyc[i] ? host_cyc[i] : 1);
  *result = acc / sms;
  return cudaSuccess;
}

}  // namespace fa
