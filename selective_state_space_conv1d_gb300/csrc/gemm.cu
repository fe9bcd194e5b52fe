// gemm.cu - the projections of the Mamba-1 layer (in_proj, x_proj, dt_proj,
// out_proj) as one bf16 tensor-core GEMM for sm_103a:
//
//   C[M][N] = A[M][K] . W[N][K]^T  (+ R[M][N])      f32 accumulation
//
// A and W are bf16, row-major with K contiguous (a linear layer's activations
// and its [out_features][in_features] weight); C is f32 or bf16; R, the
// residual, f32.  (mamba-rs inference.rs step chain F2 in_proj, F5 x_proj, F6
// dt_proj, F11 out_proj + residual; prefill.rs `prefill_body` runs the same
// projections over all T rows.)
//
// Design (one CTA per 128 x BN output tile, 4 warps):
//  * TMA (cp.async.bulk.tensor.2d, 128-byte swizzle) brings 128 x 64 tiles of
//    A and BN x 64 tiles of W into a 3-stage shared-memory ring; an mbarrier
//    per stage says "landed" (transaction bytes) and another "consumed".
//    Rows and columns past M, N or K are zero-filled by the TMA unit.
//  * One thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> f32, M 128,
//    N BN, K 16 per instruction) from the shared-memory descriptors into a
//    BN-column accumulator in tensor memory; tcgen05.commit frees a stage when
//    its MMAs are done, and a last commit tells the epilogue.
//  * The four warps read the accumulator back (tcgen05.ld, 32 lanes x 32 bit,
//    warp w owning rows 32w..32w+31) into shared memory (the ring is free by
//    then), and the CTA stores it row by row with 16-byte coalesced accesses,
//    adding the residual and rounding on the way.
//  * Every mbarrier wait is bounded (about a second); one that runs out sets
//    MAMBA_FAULT_GEMM_WAIT, and the CTA still waits (bounded) for its copies and
//    MMAs in flight and frees its tensor memory before it returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/mamba_ssm.h"
#include "async_copy.cuh"
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kBM = 128;        // rows per tile (the MMA's M)
constexpr int kBK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 3;  // two CTAs per SM: one's epilogue overlaps the other's main loop
constexpr int kThreads = 128;
constexpr long long kWaitLimit = 1ll << 31;  // SM cycles (about a second)

__device__ int g_gemm_faults = 0;

template <int BN>
struct GemmSmem {
  static constexpr int kA = kBM * kBK * 2;  // bytes per stage
  static constexpr int kB = BN * kBK * 2;
  static constexpr int kStage = kA + kB;
  static constexpr int kRing = kStages * kStage;
  static constexpr int kPitch = BN + 4;                  // epilogue staging row, floats (bank-conflict free)
  static constexpr int kStaged = kBM * kPitch * 4;       // the staged accumulator reuses the ring
  static constexpr int kBar = kRing > kStaged ? kRing : kStaged;  // mbarriers after both
  static constexpr int kBytes = kBar + 8 * (2 * kStages + 1) + 16;
  static constexpr int kAlloc = kBytes + 1024;           // room to align the base to 1024 bytes
};

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 64 bf16 (128 bytes), 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;              // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: 8 rows x 128 bytes
  d |= (uint64_t)1 << 46;              // descriptor version of sm_100 and later
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: f32 accumulator, bf16 A and B, both
// K-major, N = BN, M = 128.
template <int BN>
__host__ __device__ constexpr uint32_t instr_desc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

template <int BN, bool C_BF16>
__global__ void __launch_bounds__(kThreads, 2)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w, void* c,
                     int64_t ld_c, const float* r, int64_t ld_r, int M, int N, int K, int vec_ok) {
  using L = GemmSmem<BN>;
  extern __shared__ unsigned char smem_raw[];
  grid_dependency_wait();
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;  // 1024-byte aligned for the 128-byte swizzle
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + L::kBar;
  auto full = [&](int s) { return bars + 8 * s; };
  auto empty = [&](int s) { return bars + 8 * (kStages + s); };
  const uint32_t done = bars + 8 * (2 * kStages);
  const uint32_t tmem_slot = done + 8;
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(gbase + L::kBar + 8 * (2 * kStages + 1));

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * BN;
  const int k_tiles = (K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    mbar_fence_init();
  }
  if (warp == 0) {  // the accumulator: BN columns of tensor memory
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot), "r"(BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_ptr;
  bool ok = true;

  if (warp == 0 && lane == 0) {
    // producer: TMA into the ring
    int issued = 0;
    for (int kt = 0; kt < k_tiles; ++kt) {
      const int s = kt % kStages;
      if (kt >= kStages && !mbar_wait(empty(s), ((kt / kStages) + 1) & 1, kWaitLimit)) {
        atomicOr(&g_gemm_faults, MAMBA_FAULT_GEMM_WAIT);
        break;
      }
      const uint32_t sa = base + s * L::kStage, sb = sa + L::kA;
      mbar_arrive_expect_tx(full(s), L::kStage);
      tma_load_2d(sa, &map_a, kt * kBK, m0, full(s));
      tma_load_2d(sb, &map_w, kt * kBK, n0, full(s));
      issued = kt + 1;
    }
    // every copy issued lands before this thread moves on
    for (int kt = issued > kStages ? issued - kStages : 0; kt < issued; ++kt)
      if (!mbar_wait(full(kt % kStages), (kt / kStages) & 1, kWaitLimit)) atomicOr(&g_gemm_faults, MAMBA_FAULT_GEMM_WAIT);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = instr_desc<BN>();
    for (int kt = 0; kt < k_tiles; ++kt) {
      const int s = kt % kStages;
      if (!mbar_wait(full(s), (kt / kStages) & 1, kWaitLimit)) {
        atomicOr(&g_gemm_faults, MAMBA_FAULT_GEMM_WAIT);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t sa = base + s * L::kStage, sb = sa + L::kA;
      const uint64_t da = smem_desc(sa), db = smem_desc(sb);
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k)  // 16 bf16 = 32 bytes = 2 descriptor units per step
        mma_bf16(tmem, da + 2 * k, db + 2 * k, idesc, (kt > 0 || k > 0) ? 1u : 0u);
      mma_commit(empty(s));
    }
    mma_commit(done);  // also after a failed wait: the epilogue waits for the MMAs in flight
  }
  __syncwarp();

  // epilogue: all four warps; warp w reads accumulator lanes (rows) 32w..32w+31
  if (!mbar_wait(done, 0, kWaitLimit)) {
    if (lane == 0) atomicOr(&g_gemm_faults, MAMBA_FAULT_GEMM_WAIT);
    ok = false;
  }
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  float* stage_f = reinterpret_cast<float*>(gbase);  // [kBM][kPitch], over the (now idle) ring
  if (ok) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      uint32_t v[16];
      const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0;
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
          "%15}, [%16];"
          : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
            "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
          : "r"(taddr)
          : "memory");
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      float4* dst = reinterpret_cast<float4*>(stage_f + (warp * 32 + lane) * L::kPitch + c0);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                             __uint_as_float(v[4 * j + 3]));
    }
  }
  __syncthreads();
  if (ok) {
    // row by row: 4 consecutive columns per thread, BN / 4 threads per row
    constexpr int kTPR = BN / 4;
    constexpr int kRowsPer = kThreads / kTPR;
    const int cq = (threadIdx.x % kTPR) * 4;
    const int col = n0 + cq;
    // vec_ok: c (and r) aligned for 4-column vector accesses, strides multiples of 4
    const bool vec = vec_ok && col + 3 < N;
#pragma unroll 1
    for (int rr = threadIdx.x / kTPR; rr < kBM; rr += kRowsPer) {
      const int row = m0 + rr;
      if (row >= M) break;
      float4 x = *reinterpret_cast<const float4*>(stage_f + rr * L::kPitch + cq);
      float xs[4] = {x.x, x.y, x.z, x.w};
      if (vec) {
        if (r) {
          const float4 rv = *reinterpret_cast<const float4*>(r + (int64_t)row * ld_r + col);
          xs[0] += rv.x; xs[1] += rv.y; xs[2] += rv.z; xs[3] += rv.w;
        }
        if (C_BF16) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(xs[0], xs[1]), hi = __floats2bfloat162_rn(xs[2], xs[3]);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(c) + (int64_t)row * ld_c + col) = pk;
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(c) + (int64_t)row * ld_c + col) =
              make_float4(xs[0], xs[1], xs[2], xs[3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (col + j >= N) break;
          float xv = xs[j];
          if (r) xv += r[(int64_t)row * ld_r + col + j];
          if (C_BF16)
            reinterpret_cast<__nv_bfloat16*>(c)[(int64_t)row * ld_c + col + j] = __float2bfloat16_rn(xv);
          else
            reinterpret_cast<float*>(c)[(int64_t)row * ld_c + col + j] = xv;
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  grid_dependents_launch();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BN) : "memory");
}

// cuTensorMapEncodeTiled from the driver, looked up once
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
      cudaGetLastError();
      return nullptr;
    }
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// A 2-D tensor map over rows x cols bf16 (row stride ld elements), boxes of
// box_rows x 64 with 128-byte swizzle; out-of-range elements read as zero.
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool C_BF16>
cudaError_t launch_bn(const GemmArgs& g, const CUtensorMap& ma, const CUtensorMap& mw, cudaStream_t stream) {
  auto kern = gemm_bf16_kernel<BN, C_BF16>;
  static int configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!__atomic_load_n(&configured[dev], __ATOMIC_RELAXED)) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmSmem<BN>::kAlloc)) !=
        cudaSuccess)
      return e;
    __atomic_store_n(&configured[dev], 1, __ATOMIC_RELAXED);
  }
  const dim3 grid((unsigned)((g.M + kBM - 1) / kBM), (unsigned)((g.N + BN - 1) / BN));
  const uintptr_t cp = reinterpret_cast<uintptr_t>(g.c), rp = reinterpret_cast<uintptr_t>(g.r);
  const int vec_ok = (cp % (C_BF16 ? 8 : 16)) == 0 && g.ld_c % 4 == 0 && (!g.r || (rp % 16 == 0 && g.ld_r % 4 == 0));
  return launch_pdl(false, kern, grid, dim3(kThreads), (size_t)GemmSmem<BN>::kAlloc, stream, ma, mw, g.c, g.ld_c, g.r,
                    g.ld_r, (int)g.M, (int)g.N, (int)g.K, vec_ok);
}

}  // namespace

cudaError_t launch_gemm_bf16(const GemmArgs& g, cudaStream_t stream) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  // output tiles of 128 x BN: narrow outputs (x_proj's dt_rank + 2 d_state)
  // take BN = 64, the rest 128
  const int bn = g.N <= 64 ? 64 : 128;
  CUtensorMap ma, mw;
  if (!make_map(&ma, g.a, g.M, g.K, g.ld_a, kBM) || !make_map(&mw, g.w, g.N, g.K, g.ld_w, bn))
    return cudaErrorInvalidValue;
  if (bn == 64) return g.c_bf16 ? launch_bn<64, true>(g, ma, mw, stream) : launch_bn<64, false>(g, ma, mw, stream);
  return g.c_bf16 ? launch_bn<128, true>(g, ma, mw, stream) : launch_bn<128, false>(g, ma, mw, stream);
}

int read_gemm_faults(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_faults, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_gemm_faults, &zero, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace mamba
