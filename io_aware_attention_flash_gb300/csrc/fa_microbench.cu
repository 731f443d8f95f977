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
// cvt.rn.bf16x2.f32; 4: two ex2 and a bf16 pack by integer rounding (add
// 0x8000, keep the high halves); 5: the forward softmax's full step (paired
// FMA, two ex2, paired add into a row sum, cvt pack); 6: kind 5 with the
// integer pack of kind 4; 7: kind 5 with a quarter of the pairs through the
// polynomial exp2 (ex2_poly2) instead of the special-function unit.
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
        uint32_t pk;
        if constexpr (KIND == 3 || KIND == 5 || KIND == 7)
          pk = pack_bf16x2(a, b);
        else
          pk = __byte_perm(__float_as_uint(a) + 0x8000u, __float_as_uint(b) + 0x8000u, 0x7632);
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

// The forward kernel's softmax on one 128 x 128 score tile, alone: no MMA
// runs.  Warpgroup t (t < NWG) reads S_t (128 columns of TMEM, random fp32
// scores), takes the row max, forms P = 2^(c·s − c·m) with the paired FMA,
// ex2, the paired row-sum adds and the bf16 packing, and stores P (64
// columns) into a separate TMEM region, as the kernel does, `iters` times.
// Cycles per tile show whether the softmax's instruction stream or its
// surroundings in the kernel set its duration.
template <int NWG>
__global__ void __launch_bounds__(320, 1) softmax_tile_kernel(int iters, unsigned long long* cycles, float* sink) {
  // (register budget of the forward kernel's 320 threads)
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x / 32;
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int t = warp / 4, wq = warp % 4;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const uint32_t tS = lane_addr + 128 * t, tP = lane_addr + 256 + 64 * t;
  {
    uint32_t z[32];
    for (int cc = 0; cc < 128; cc += 32) {
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = __float_as_uint(-4.0f + 8.0f * ((random_bf16x2(threadIdx.x * 131 + cc + i) & 0xFFFFu) / 65536.0f));
      tmem_st32(tS + cc, z);
    }
    tmem_wait_st();
  }
  __syncthreads();
  const float c = 0.1275f;
  float l = 0.f;
  const unsigned long long t0 = clock64();
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
    uint32_t s[4][32];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) tmem_ld32(tS + ch * 32, s[ch]);
    tmem_wait_ld();
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) reg_fence(s[ch]);
    float mx[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) mx[k] = -CUDART_INF_F;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        mx[i & 3] = fmax3(mx[i & 3], __uint_as_float(s[ch][2 * i]), __uint_as_float(s[ch][2 * i + 1]));
    const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    const float mc = mt * c;
    const uint64_t c2 = f2_pack(c, c), nmc2 = f2_pack(-mc, -mc);
    uint64_t ls2[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ls2[k] = f2_pack(0.f, 0.f);
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float x0, x1;
        f2_unpack(ffma2(f2_pack(__uint_as_float(s[ch][2 * e]), __uint_as_float(s[ch][2 * e + 1])), c2, nmc2), x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        ls2[e & 3] = fadd2(ls2[e & 3], f2_pack(p0, p1));
        pk[e] = pack_bf16x2(p0, p1);
      }
      tmem_st16(tP + ch * 16, pk);
    }
    float ls[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) f2_unpack(ls2[k], ls[2 * k], ls[2 * k + 1]);
    l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
    tmem_wait_st();
  }
  const unsigned long long t1 = clock64();
  if (l == 12345.f) sink[threadIdx.x % kMaxSms] = l;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
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
// other unit holds it up.  With BUSY, two more warps on the issuing warp's
// SM sub-partition run an FMA / ex2 mix (as softmax warps do) until the MMA
// loop ends, so the rate shows what sharing the sub-partition's issue slots
// costs the issuing thread.  The operand descriptors are formed as in the
// forward kernel (tile bases once, a 64-bit add per K step).  COMMITS = 2
// adds a tcgen05.commit (to an mbarrier nobody waits on) after each S_t, as
// the forward kernel signals each S_t to its softmax; COMMITS = 4 adds one
// after each PV_t too.  WAITS adds, per iteration, the forward kernel's four
// mbarrier waits (V, K and P_0 before PV_0, P_1 before PV_1) on an mbarrier
// whose phase has already completed; RING takes the K and V operands from
// 3- and 2-slot rings indexed by the iteration, as the forward kernel does.
template <int DPV, bool ALIAS, bool SPLIT, bool BUSY = false, int GAP = 0, int COMMITS = 0, bool WAITS = false,
          bool RING = false>
__global__ void __launch_bounds__(384, 1) fwd_stream_kernel(int iters, unsigned long long* cycles, uint32_t* err) {
  static_assert(ALIAS || DPV == 64, "separate P columns fit only beside 64-column O tiles");
  constexpr int TILE = 128 * 128 * 2;  // one 128 x 128 bf16 tile: two 128-byte swizzled 64-column blocks
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ __align__(8) uint64_t sink_bar;
  __shared__ __align__(8) uint64_t ready_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int mma_done;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gen = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) mma_done = 0;
  for (int i = threadIdx.x; i < 3 * TILE / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gen)[i] =
        make_uint4(random_bf16x2(4 * i), random_bf16x2(4 * i + 1), random_bf16x2(4 * i + 2), random_bf16x2(4 * i + 3));
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done_bar), 1);
    mbar_init(smem_u32(&sink_bar), 1);
    mbar_init(smem_u32(&ready_bar), 1);
    fence_mbar_init();
    mbar_arrive(smem_u32(&ready_bar));  // phase 0 complete: every wait below passes
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
    const uint32_t ready = smem_u32(&ready_bar);
    auto wait_ready = [&]() {
      if (WAITS) {
        wait_bounded(ready, 0, &mma_done, err, 1000000000ull);
        tc_fence_after();
      }
    };
    const uint64_t dK_ring0 = dQ, dV_ring0 = sdesc_sw128(sK, 128 * 128, 1024);
    int ks = 0, vs = 0;
    const unsigned long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
      if (SPLIT) {
        pv(0); pv(1); sg(0); sg(1);
      } else if (COMMITS > 0) {
        const uint32_t sink = smem_u32(&sink_bar);
        if (RING) {  // K slots: the three tiles; V slots: the last two
          dKi = sdesc_add(dK_ring0, ks * TILE);
          dVi = sdesc_add(dV_ring0, vs * TILE);
          if (++ks == 3) ks = 0;
          if (++vs == 2) vs = 0;
        }
        wait_ready();
        wait_ready();
        wait_ready();
        pv(0);
        if (COMMITS >= 4) tc_commit(sink);
        sg(0);
        tc_commit(sink);
        wait_ready();
        pv(1);
        if (COMMITS >= 4) tc_commit(sink);
        sg(1);
        tc_commit(sink);
      } else {
        pv(0); sg(0); pv(1); sg(1);
      }
      if (GAP > 0) {  // the issuing thread idles GAP cycles once per iteration
        const long long tg = clock64();
        while (clock64() - tg < GAP) {
        }
      }
    }
    tc_commit(smem_u32(&done_bar));
    wait_drain(smem_u32(&done_bar), 0, err, 2000000000ull);
    const unsigned long long t1 = clock64();
    cycles[blockIdx.x] = t1 - t0;
    mma_done = 1;
  } else if (BUSY && (warp == 4 || warp == 8)) {
    // Softmax-like issue load on sub-partition 0: FMA, ex2 and add per element,
    // until the MMA loop is done (and at most 2^22 rounds).
    float x[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = -1.0f - 0.001f * (threadIdx.x + c);
    for (int it = 0; it < (1 << 22) && !mma_done; ++it) {
#pragma unroll
      for (int c = 0; c < 8; ++c) x[c] = ex2_approx(fmaf(x[c], 0.999f, -0.001f)) - 1.5f;
    }
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) acc += x[c];
    if (acc == 12345.f) cycles[blockIdx.x] = 0;  // keeps the loop alive
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DPV, bool ALIAS, bool SPLIT, bool BUSY = false, int GAP = 0, int COMMITS = 0, bool WAITS = false,
          bool RING = false>
cudaError_t launch_fwd_stream(int sms, int iters, unsigned long long* cyc, uint32_t* err, cudaStream_t s) {
  const int smem = 3 * 128 * 128 * 2 + 1024;
  auto kern = fwd_stream_kernel<DPV, ALIAS, SPLIT, BUSY, GAP, COMMITS, WAITS, RING>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<sms, BUSY ? 384 : 128, smem, s>>>(iters, cyc, err);
  return cudaGetLastError();
}

// Reduce-add throughput into a global fp32 array shaped like the backward's
// dQ accumulator ([rows, 16, 128]), from a CTA of 8 warps per SM.  Each warp
// repeatedly adds a 32-row x 32-column fp32 chunk at a pseudo-random place:
//   VIA_TMA: stages the chunk in its own 4 KB shared-memory slot (NSLOT slots
//            per warp, used in turn) and issues one TMA bulk reduce-add, as
//            the backward's dQ drain does;
//   MODE 1:  each lane adds its row's 128 bytes from registers with eight
//            16-byte vector atomics (a warp instruction touches 32 rows);
//   MODE 2:  the same atomics laid out so that one warp instruction covers
//            512 contiguous bytes (the array read as 128-row tiles, a 16-byte
//            column chunk of 128 consecutive rows stored together);
//   MODE 3:  warps 0-3 as VIA_TMA, warps 4-7 as MODE 2 (both paths at once).
// Reports bytes added per SM per clock.
template <bool VIA_TMA, int NSLOT, int MODE = 0>
__global__ void __launch_bounds__(256, 1)
    reduce_rate_kernel(const __grid_constant__ CUtensorMap tm, float* buf, int rows, int iters,
                       unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int ntile = rows / 32;
  uint32_t v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(1e-7f * (lane + i));
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    const int c0 = 32 * (warp & 3);
    const int h = (blockIdx.x + it) & 15;
    const int row = ((blockIdx.x * 131 + it * 7 + (warp >> 2) * 3) % ntile) * 32;
    const bool use_tma = VIA_TMA || (MODE == 3 && warp < 4);
    if (use_tma) {
      const uint32_t slot = base + (warp * NSLOT + it % NSLOT) * 4096;
      if (it >= NSLOT) {
        if (lane == 0) bulk_wait_group_read<NSLOT - 1>();
        __syncwarp();
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t chunk = u ^ (lane & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(slot + lane * 128 + chunk * 16), "r"(v[4 * u]),
                     "r"(v[4 * u + 1]), "r"(v[4 * u + 2]), "r"(v[4 * u + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_3d(&tm, slot, c0, h, row);
        bulk_commit_group();
      }
    } else if (MODE == 1) {
      float* dst = buf + (static_cast<size_t>(row + lane) * 16 + h) * 128 + c0;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        atomicAdd(reinterpret_cast<float4*>(dst + 4 * u),
                  make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]), __uint_as_float(v[4 * u + 2]),
                              __uint_as_float(v[4 * u + 3])));
    } else {
      // 128-row tile (row / 128, h), 16-byte column chunk k: 128 rows x 16 B contiguous
      const int R = row + lane;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = c0 / 4 + u;
        float* dst = buf + ((static_cast<size_t>(R >> 7) * 16 + h) * 32 + k) * 512 + (R & 127) * 4;
        atomicAdd(reinterpret_cast<float4*>(dst),
                  make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]), __uint_as_float(v[4 * u + 2]),
                              __uint_as_float(v[4 * u + 3])));
      }
    }
  }
  if (VIA_TMA || MODE == 3) {
    if (lane == 0) bulk_wait_group0();
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <bool VIA_TMA, int NSLOT, int MODE = 0>
cudaError_t launch_reduce_rate(int sms, const CUtensorMap& tm, float* buf, int rows, int iters,
                               unsigned long long* cyc, cudaStream_t s) {
  const int smem = (VIA_TMA || MODE == 3) ? 8 * NSLOT * 4096 + 1024 : 0;
  cudaError_t e = cudaFuncSetAttribute(reduce_rate_kernel<VIA_TMA, NSLOT, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  reduce_rate_kernel<VIA_TMA, NSLOT, MODE><<<sms, 256, smem, s>>>(tm, buf, rows, iters, cyc);
  return cudaGetLastError();
}

}  // namespace

// Runs one microbenchmark with one CTA per SM and returns the mean over CTAs
// of (units retired by the CTA) / (its SM cycles).
// Cycles one thread spends on one synchronisation step, timed with the SM
// cycle counter around the step and a branch on its result (as a waiting
// thread consumes it).  KIND 0: mbarrier.try_wait on a completed phase;
// 1: the same plus tcgen05.fence::after_thread_sync; 2: mbarrier.test_wait on
// a completed phase; 3: a volatile shared-memory load of a flag;
// 4: tcgen05.commit; 5: tcgen05.fence::after_thread_sync alone; 6: nothing
// (the timer's own cost).  With FULL the thread first issues 16 MMAs of the
// forward kernel's shape, so the step runs while the tensor pipe's queue is
// full, as it does in the forward kernel's MMA thread.
template <int KIND, bool FULL>
__global__ void __launch_bounds__(128, 1) sync_latency_kernel(int iters, unsigned long long* cycles, uint32_t* err) {
  constexpr int TILE = 128 * 128 * 2;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t ready_bar, sink_bar, done_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gen = smem_raw + (base - raw);
  for (int i = threadIdx.x; i < 2 * TILE / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(gen)[i] =
        make_uint4(random_bf16x2(4 * i), random_bf16x2(4 * i + 1), random_bf16x2(4 * i + 2), random_bf16x2(4 * i + 3));
  if (threadIdx.x == 0) {
    flag = 1;
    mbar_init(smem_u32(&ready_bar), 1);
    mbar_init(smem_u32(&sink_bar), 1);
    mbar_init(smem_u32(&done_bar), 1);
    fence_mbar_init();
    mbar_arrive(smem_u32(&ready_bar));
  }
  fence_proxy_async_smem();
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    const uint64_t dQ = sdesc_sw128(base, 16, 1024), dK = sdesc_sw128(base + TILE, 16, 1024);
    const uint32_t ready = smem_u32(&ready_bar), sink = smem_u32(&sink_bar), done = smem_u32(&done_bar);
    unsigned long long total = 0;
    uint32_t bad = 0, phase = 0;
    for (int i = 0; i < iters; ++i) {
      if (FULL) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint32_t koff = ((kk % 8) / 4) * (128 * 128) + (kk % 4) * 32;
          mma_ss(tmem + 128 * (kk / 8), sdesc_add(dQ, koff), sdesc_add(dK, koff), idesc_s, (kk % 8) > 0 ? 1u : 0u);
        }
      }
      const long long t0 = clock64();
      if constexpr (KIND == 0 || KIND == 1) {
        if (!mbar_try_wait(ready, 0)) ++bad;
        if (KIND == 1) tc_fence_after();
      } else if constexpr (KIND == 2) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(ready), "r"(0u)
            : "memory");
        if (!ok) ++bad;
      } else if constexpr (KIND == 3) {
        if (flag != 1) ++bad;
      } else if constexpr (KIND == 4) {
        tc_commit(sink);
      } else if constexpr (KIND == 5) {
        tc_fence_after();
      }
      const long long t1 = clock64();
      total += t1 - t0;
      if (FULL) {
        tc_commit(done);
        if (!wait_drain(done, phase, err, 1000000000ull)) break;
        phase ^= 1;
      }
    }
    cycles[blockIdx.x] = total + (bad ? 1000000000ull : 0ull);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int KIND, bool FULL>
cudaError_t launch_sync_latency(int sms, int iters, unsigned long long* cyc, uint32_t* err, cudaStream_t s) {
  const int smem = 2 * 128 * 128 * 2 + 1024;
  auto kern = sync_latency_kernel<KIND, FULL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<sms, 128, smem, s>>>(iters, cyc, err);
  return cudaGetLastError();
}

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
    case 39: unit_rate_kernel<4><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 40: unit_rate_kernel<5><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 41: unit_rate_kernel<6><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 43: unit_rate_kernel<7><<<sms, threads, 0, s>>>(iters, cyc, sink); break;
    case 44: softmax_tile_kernel<1><<<sms, 128, 0, s>>>(iters, cyc, sink); break;
    case 45: softmax_tile_kernel<2><<<sms, 256, 0, s>>>(iters, cyc, sink); break;
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
    case 17: e = launch_fwd_stream<128, true, false, true>(sms, iters, cyc, err, s); break;
    case 18: e = launch_fwd_stream<128, true, false, false, 256>(sms, iters, cyc, err, s); break;
    case 19: e = launch_fwd_stream<128, true, false, false, 600>(sms, iters, cyc, err, s); break;
    case 20: e = launch_fwd_stream<128, true, false, false, 1200>(sms, iters, cyc, err, s); break;
    case 21: e = launch_fwd_stream<128, true, false, false, 0, 2>(sms, iters, cyc, err, s); break;
    case 22: e = launch_fwd_stream<128, true, false, false, 0, 4>(sms, iters, cyc, err, s); break;
    case 23: e = launch_fwd_stream<128, true, false, false, 0, 4, true>(sms, iters, cyc, err, s); break;
    case 24: e = launch_fwd_stream<128, true, false, false, 0, 4, true, true>(sms, iters, cyc, err, s); break;
    case 25: e = launch_sync_latency<0, false>(sms, iters, cyc, err, s); break;
    case 26: e = launch_sync_latency<1, false>(sms, iters, cyc, err, s); break;
    case 27: e = launch_sync_latency<2, false>(sms, iters, cyc, err, s); break;
    case 28: e = launch_sync_latency<3, false>(sms, iters, cyc, err, s); break;
    case 29: e = launch_sync_latency<4, false>(sms, iters, cyc, err, s); break;
    case 30: e = launch_sync_latency<6, false>(sms, iters, cyc, err, s); break;
    case 31: e = launch_sync_latency<0, true>(sms, iters, cyc, err, s); break;
    case 32: e = launch_sync_latency<1, true>(sms, iters, cyc, err, s); break;
    case 33: e = launch_sync_latency<2, true>(sms, iters, cyc, err, s); break;
    case 34: e = launch_sync_latency<3, true>(sms, iters, cyc, err, s); break;
    case 35: e = launch_sync_latency<4, true>(sms, iters, cyc, err, s); break;
    case 36: e = launch_sync_latency<5, true>(sms, iters, cyc, err, s); break;
    case 37: e = launch_sync_latency<6, true>(sms, iters, cyc, err, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if (which <= 2)
    units_per_cta = static_cast<double>(threads) * iters * kChains;
  else if (which >= 38)  // two exponentials per step (38-41, 43)
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
  if ((which >= 25 && which <= 37) || which == 44 || which == 45) {  // cycles per step, averaged over the SMs
    for (int i = 0; i < sms; ++i) acc += static_cast<double>(host_cyc[i]) / iters;
    *result = acc / sms;
    return cudaSuccess;
  }
  for (int i = 0; i < sms; ++i) acc += units_per_cta / static_cast<double>(host_cyc[i] ? host_cyc[i] : 1);
  *result = acc / sms;
  return cudaSuccess;
}

// Reduce-add throughput (see reduce_rate_kernel); `tm` maps `buf` as
// [rows, 16, 128] fp32 with a 32 x 1 x 32 box.  which = 12: TMA, one slot per
// warp; 13: TMA, two slots per warp; 14: vector atomics, 32 rows per warp
// instruction; 15: vector atomics, 512 contiguous bytes per warp instruction;
// 16: TMA and contiguous atomics from half the warps each.
cudaError_t run_reduce_microbench(int which, int iters, const CUtensorMap& tm, float* buf, int rows, double* result,
                                  cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (sms > kMaxSms) sms = kMaxSms;
  unsigned long long* cyc = nullptr;
  if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&cyc), g_cycles)) != cudaSuccess) return e;
  switch (which) {
    case 12: e = launch_reduce_rate<true, 1>(sms, tm, buf, rows, iters, cyc, s); break;
    case 13: e = launch_reduce_rate<true, 2>(sms, tm, buf, rows, iters, cyc, s); break;
    case 14: e = launch_reduce_rate<false, 1, 1>(sms, tm, buf, rows, iters, cyc, s); break;
    case 15: e = launch_reduce_rate<false, 1, 2>(sms, tm, buf, rows, iters, cyc, s); break;
    case 16: e = launch_reduce_rate<false, 1, 3>(sms, tm, buf, rows, iters, cyc, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  static unsigned long long host_cyc[kMaxSms];
  if ((e = cudaMemcpy(host_cyc, cyc, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return e;
  const double bytes_per_cta = 8.0 * 4096.0 * iters;
  double acc = 0;
  for (int i = 0; i < sms; ++i) acc += bytes_per_cta / static_cast<double>(host_cyc[i] ? host_cyc[i] : 1);
  *result = acc / sms;
  return cudaSuccess;
}

}  // namespace fa
