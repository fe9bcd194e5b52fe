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
// Design (persistent: one CTA per SM, tiles of 128 x BN, BN 64 / 128 / 192 / 256):
//  * TMA (cp.async.bulk.tensor.2d, 128-byte swizzle) brings 128 x 64 tiles of
//    A and BN x 64 tiles of W into a shared-memory ring of 4-8 stages; an
//    mbarrier per stage says "landed" (transaction bytes) and another
//    "consumed".  Rows and columns past M, N or K are zero-filled by TMA.
//  * One thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> f32, M 128,
//    N BN, K 16 per instruction) from the shared-memory descriptors into one
//    of two BN-column accumulators in tensor memory; tcgen05.commit frees a
//    stage when its MMAs are done, and marks the accumulator full at the end
//    of a tile.
//  * Four epilogue warps drain the other accumulator meanwhile (tcgen05.ld,
//    32 lanes x 32 columns, warp w owning tile rows 32 (w % 4) ...).  A bf16
//    output is packed into 32 x 64 boxes in the 128-byte swizzled layout and
//    leaves by tensor stores (cp.async.bulk.tensor, clipped at M and N); an
//    f32 output stages 32 x 32 blocks and stores them with 16-byte coalesced
//    accesses, adding the residual on the way.  A wide tile reads half the
//    shared memory per MMA of a 128-wide one; the double accumulator hides
//    the epilogue behind the next tile's MMAs.
//  * Few output tiles and a long K (the decode projections): K is split over a
//    thread-block cluster whose ranks reduce through distributed shared memory
//    (see the kernel's comment).
//  * Every mbarrier wait is bounded (about a second); one that runs out sets
//    MAMBA_FAULT_GEMM_WAIT and an abort flag that ends every role's loop; the
//    CTA still waits (bounded) for its copies and MMAs in flight and frees its
//    tensor memory before it returns.
#include <cooperative_groups.h>
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
constexpr int kThreads = 192;   // warp 0 TMA, warp 1 MMA (and tensor-memory owner), warps 2-5 epilogue
constexpr int kEpiWarps = 4;
constexpr int kChunk = 32;      // epilogue columns per tensor-memory load
constexpr int kStagePitch = kChunk + 4;  // floats per staged row (16-byte rows, conflict-free)
constexpr int kSmemLimit = 232448;       // opt-in shared memory per block on sm_103a
constexpr long long kWaitLimit = 1ll << 31;  // SM cycles (about a second)

__device__ int g_gemm_faults = 0;

template <int BN, int MAX_STAGES = 8>
struct GemmSmem {
  static constexpr int kA = kBM * kBK * 2;  // bytes per stage
  static constexpr int kB = BN * kBK * 2;
  static constexpr int kStage = kA + kB;
  // epilogue staging per warp: 32 rows of 32 f32 (padded), or two 4 KB bf16
  // buffers for the tensor-memory-accelerator stores; 1024-byte aligned
  static constexpr int kEpiF32 = kEpiWarps * 32 * kStagePitch * 4;
  static constexpr int kEpiTma = kEpiWarps * 2 * 4096;
  static constexpr int kEpi = kEpiF32 > kEpiTma ? kEpiF32 : kEpiTma;
  static constexpr int kFixed = kEpi + 256 + 1024;  // staging, barriers, base alignment
  static constexpr int kStages0 = (kSmemLimit - kFixed) / kStage;
  static constexpr int kStages = kStages0 > MAX_STAGES ? MAX_STAGES : kStages0;
  static constexpr int kRing = kStages * kStage;
  static constexpr int kBar = kRing + kEpi;                 // barriers after the ring and the staging
  static constexpr int kBytes = kBar + 8 * (2 * kStages + 5) + 16;
  static constexpr int kAlloc = kBytes + 1024;              // room to align the base to 1024 bytes
  // accumulator a starts at column a * kAccCols: BN rounded up to a power of
  // two, so each accumulator starts on a boundary of its own width
  static constexpr int kAccCols = BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static constexpr int kTmemCols = 2 * kAccCols;
  static_assert(kStages >= 2, "shared memory too small for two stages");
  static_assert(kAlloc <= kSmemLimit, "shared memory over the opt-in limit");
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

// the same with an L2 eviction-priority hint (a createpolicy value)
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
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

// shared -> global tensor store of one box, in a bulk group
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
               "r"(y), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most N of this thread's bulk groups still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy shared-memory writes visible to the tensor memory accelerator
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// distributed shared memory: this CTA's shared address in cluster rank `rank`,
// and a 16-byte load from there
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 dsmem_ld4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 lanes x 32 columns of f32 from tensor memory, asynchronous: the registers
// may be read only after tmem_wait on the same array.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// Waits for this thread's tensor-memory loads; the registers are threaded
// through so that no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_wait(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                 "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                 "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                 "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// One 32 x 32 block of the accumulator, held one row per lane in v, to C:
// staged through this warp's shared memory and stored 4 rows x 32 columns per
// step (8 lanes x 4 columns per row), the residual added and the value rounded
// on the way.  full: the block is inside M and N and the vector accesses are
// aligned -- then the 8 residual loads are issued together, branch-free.
template <bool C_BF16>
__device__ __forceinline__ void emit_block(const uint32_t (&v)[32], float* stage_f, int lane, int row0, int col0,
                                           bool full, void* c, int64_t ld_c, const float* r, int64_t ld_r, int M,
                                           int N) {
  float4* dst = reinterpret_cast<float4*>(stage_f + lane * kStagePitch);
#pragma unroll
  for (int j = 0; j < 8; ++j)
    dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                         __uint_as_float(v[4 * j + 3]));
  __syncwarp();
  const int cq = (lane & 7) * 4;
  const int col = col0 + cq;
  const int rsub = lane >> 3;
  if (full) {
    float4 rv[8];
    if (r) {
#pragma unroll
      for (int it = 0; it < 8; ++it)
        rv[it] = *reinterpret_cast<const float4*>(r + (int64_t)(row0 + it * 4 + rsub) * ld_r + col);
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int rr = it * 4 + rsub;
      float4 x = *reinterpret_cast<const float4*>(stage_f + rr * kStagePitch + cq);
      if (r) {
        x.x += rv[it].x;
        x.y += rv[it].y;
        x.z += rv[it].z;
        x.w += rv[it].w;
      }
      const int64_t off = (int64_t)(row0 + rr) * ld_c + col;
      if (C_BF16) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(c) + off) = pk;
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(c) + off) = x;
      }
    }
  } else {
    // an edge block: element by element, inside M and N only
#pragma unroll 1
    for (int it = 0; it < 8; ++it) {
      const int rr = it * 4 + rsub;
      const int row = row0 + rr;
      if (row >= M) break;
      const float* xs = stage_f + rr * kStagePitch + cq;
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
  __syncwarp();
}

// The output tile of the persistent schedule's `t`-th tile: groups of
// `group_m` row blocks sweep all column blocks, row blocks fastest, so the
// CTAs of one wave share a few weight tiles, and a group's activation rows
// (sized on the host to stay in L2) are read from DRAM once while the weight
// is read once per group.
__device__ __forceinline__ void tile_coords(int t, int m_tiles, int n_tiles, int group_m, int& mb, int& nb) {
  const int per_group = group_m * n_tiles;
  const int g = t / per_group, r = t % per_group;
  const int m0 = g * group_m;
  const int rows = m_tiles - m0 < group_m ? m_tiles - m0 : group_m;
  mb = m0 + r % rows;
  nb = r / rows;
}

__device__ __forceinline__ void fail_gemm(volatile int* abort_flag) {
  atomicOr(&g_gemm_faults, MAMBA_FAULT_GEMM_WAIT);
  *abort_flag = 1;
}

// Persistent, warp-specialised: each CTA takes tiles blockIdx.x, +gridDim.x, ...
//  * warp 0 (one lane) streams the A and W tiles of every K step of every
//    tile into a kStages-deep ring (TMA; "full" / "empty" barriers per stage);
//  * warp 1 (one lane) issues the MMAs of a tile into one of two
//    tensor-memory accumulators and commits "accumulator full";
//  * warps 2-5 drain the other accumulator meanwhile (tcgen05.ld; bf16 out
//    through swizzled staging and tensor stores, f32 out with its residual
//    through padded staging and 16-byte coalesced stores) and release it
//    ("accumulator empty").
//
// SPLIT (few output tiles, long K): a cluster of `splits` CTAs shares one
// tile, CTA rank q accumulating K steps [q k_tiles / splits, (q + 1) k_tiles /
// splits).  Every rank leaves its partial sums in its shared memory; after a
// cluster barrier rank q sums all ranks' partials, in rank order, for its
// 128 / splits rows of the tile through distributed shared memory and stores
// them -- a deterministic split with no global scratch and no second launch.
template <int BN, bool C_BF16, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
                     const __grid_constant__ CUtensorMap map_c, void* c, int64_t ld_c, const float* r, int64_t ld_r,
                     int M, int N, int K, int vec_ok, int splits, int group_m, int c_tma) {
  // a split CTA runs a few K steps of one tile: a short ring (two split CTAs
  // of a 64- or 128-wide tile fit on an SM)
  using L = GemmSmem<BN, SPLIT ? 3 : 8>;
  constexpr int S = L::kStages;
  static_assert(!SPLIT || kBM * (BN + 4) * 4 <= L::kRing, "the partial sums must fit in the ring");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023) & ~1023u;  // 1024-byte aligned for the 128-byte swizzle
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + L::kBar;
  auto full = [&](int s) { return bars + 8 * s; };
  auto empty = [&](int s) { return bars + 8 * (S + s); };
  auto acc_full = [&](int a) { return bars + 8 * (2 * S + a); };
  auto acc_empty = [&](int a) { return bars + 8 * (2 * S + 2 + a); };
  const uint32_t drain = bars + 8 * (2 * S + 4);
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(gbase + L::kBar + 8 * (2 * S + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_ptr + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m_tiles = (M + kBM - 1) / kBM, n_tiles = (N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;
  const int k_tiles = (K + kBK - 1) / kBK;
  // this CTA's tiles (t_first, + t_step, ...) and K steps [kb, ke)
  int rank = 0, t_first = blockIdx.x, t_step = gridDim.x, kb = 0, ke = k_tiles;
  if constexpr (SPLIT) {
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    t_first = blockIdx.x / splits;
    t_step = gridDim.x / splits;
    kb = rank * k_tiles / splits;
    ke = (rank + 1) * k_tiles / splits;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {  // two accumulators of BN f32 columns each
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_ptr)),
                 "r"(L::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_ptr;
  // every CTA is resident (one wave): the next kernel may start its set-up;
  // nothing below touches global memory before the previous kernel is done
  grid_dependents_launch();
  grid_dependency_wait();

  bool have_acc = false;  // SPLIT: this epilogue warp saw its accumulator complete
  if (warp == 0) {
    if (lane == 0) {
      // producer: TMA into the ring, K steps of all this CTA's tiles in order
      const uint64_t w_policy = l2_evict_last_policy();
      int g = 0;
      for (int t = t_first; t < tiles && !*abort_flag; t += t_step) {
        int mb, nb;
        tile_coords(t, m_tiles, n_tiles, group_m, mb, nb);
        for (int kt = kb; kt < ke; ++kt, ++g) {
          const int s = g % S;
          if (g >= S && !mbar_wait(empty(s), ((g / S) + 1) & 1, kWaitLimit)) {
            fail_gemm(abort_flag);
            break;
          }
          const uint32_t sa = base + s * L::kStage, sb = sa + L::kA;
          mbar_arrive_expect_tx(full(s), L::kStage);
          tma_load_2d(sa, &map_a, kt * kBK, mb * kBM, full(s));
          // the weight is re-read by every row-block group: keep it in L2
          tma_load_2d_hint(sb, &map_w, kt * kBK, nb * BN, full(s), w_policy);
        }
      }
      // every copy issued lands before this thread moves on
      for (int q = g > S ? g - S : 0; q < g; ++q)
        if (!mbar_wait(full(q % S), (q / S) & 1, kWaitLimit)) fail_gemm(abort_flag);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer
      constexpr uint32_t idesc = instr_desc<BN>();
      int g = 0, i = 0;
      for (int t = t_first; t < tiles && !*abort_flag; t += t_step, ++i) {
        const int a = i & 1;
        if (i >= 2 && !mbar_wait(acc_empty(a), ((i >> 1) + 1) & 1, kWaitLimit)) {
          fail_gemm(abort_flag);
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + (uint32_t)(a * L::kAccCols);
        bool ok = true;
        for (int kt = kb; kt < ke; ++kt, ++g) {
          const int s = g % S;
          if (!mbar_wait(full(s), (g / S) & 1, kWaitLimit)) {
            fail_gemm(abort_flag);
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t sa = base + s * L::kStage, sb = sa + L::kA;
          const uint64_t da = smem_desc(sa), db = smem_desc(sb);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)  // 16 bf16 = 32 bytes = 2 descriptor units per step
            mma_bf16(d, da + 2 * k, db + 2 * k, idesc, (kt > kb || k > 0) ? 1u : 0u);
          mma_commit(empty(s));
        }
        if (!ok) break;
        mma_commit(acc_full(a));
      }
      // the MMAs in flight complete before the accumulators are freed
      mma_commit(drain);
      if (!mbar_wait(drain, 0, kWaitLimit)) fail_gemm(abort_flag);
    }
  } else {
    // epilogue warps: warp w reads accumulator lanes (tile rows) 32 (w % 4) ...
    const int quad = warp & 3;
    float* stage_f = reinterpret_cast<float*>(gbase + L::kRing) + (warp - 2) * 32 * kStagePitch;
    const uint32_t tma_stage = base + L::kRing + (uint32_t)((warp - 2) * 8192);  // two 4 KB buffers
    int tma_chunk = 0;
    int i = 0;
    for (int t = t_first; t < tiles; t += t_step, ++i) {
      const int a = i & 1;
      if (*abort_flag || !mbar_wait(acc_full(a), (i >> 1) & 1, kWaitLimit)) {
        if (lane == 0 && !*abort_flag) fail_gemm(abort_flag);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if constexpr (SPLIT) {
        // one tile per CTA: every rank parks its partial sums (all BN
        // columns) in its shared memory, over the idle ring
        {
          float* part = reinterpret_cast<float*>(gbase) + (quad * 32 + lane) * (BN + 4);
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += kChunk) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, v);
            tmem_wait(v);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(part + c0 + 4 * j) =
                  make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                              __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        }
        have_acc = true;
        continue;
      }
      int mb, nb;
      tile_coords(t, m_tiles, n_tiles, group_m, mb, nb);
      const int row0 = mb * kBM + quad * 32;
      const int col0 = nb * BN;
      const int ncols = N - col0 < BN ? N - col0 : BN;  // columns of this tile inside N
      const bool rows_full = vec_ok && row0 + 32 <= M;
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(a * L::kAccCols);
      if constexpr (C_BF16) {
        if (c_tma) {
          // bf16 output through the tensor memory accelerator: 32 rows x 64
          // columns per store, staged in one of this warp's two 4 KB buffers in
          // the 128-byte swizzled layout of the box (16-byte granule j of row r
          // at granule j ^ (r % 8): conflict-free writes); the unit clips rows
          // and columns past M and N
          // (a box wholly below M is not stored at all)
#pragma unroll 1
          for (int c0 = 0; c0 < (row0 < M ? ncols : 0); c0 += 2 * kChunk, ++tma_chunk) {
            uint32_t va[32], vb[32];
            tmem_ld32(taddr + (uint32_t)c0, va);
            tmem_ld32(taddr + (uint32_t)(c0 + kChunk), vb);  // inside the accumulator even past N
            tmem_wait(va);
            tmem_wait(vb);
            const uint32_t sb = tma_stage + (uint32_t)((tma_chunk & 1) * 4096);
            if (lane == 0) bulk_wait_read<1>();  // the store two chunks back has read this buffer
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t* v = j < 4 ? va : vb;
              const int q = (j & 3) * 8;
              const uint32_t w0 = pack_bf16(v[q], v[q + 1]), w1 = pack_bf16(v[q + 2], v[q + 3]);
              const uint32_t w2 = pack_bf16(v[q + 4], v[q + 5]), w3 = pack_bf16(v[q + 6], v[q + 7]);
              const uint32_t dst = sb + (uint32_t)(lane * 128 + ((j ^ (lane & 7)) << 4));
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&map_c, col0 + c0, row0, sb);
              bulk_commit();
            }
          }
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(a));
          continue;
        }
      }
      // two blocks in flight: the next block's tensor-memory load overlaps
      // this block's stores
      uint32_t va[32], vb[32];
      tmem_ld32(taddr, va);
      tmem_wait(va);
#pragma unroll 1
      for (int c0 = 0; c0 < ncols; c0 += 2 * kChunk) {
        const bool has_b = c0 + kChunk < ncols;
        if (has_b) tmem_ld32(taddr + (uint32_t)(c0 + kChunk), vb);
        emit_block<C_BF16>(va, stage_f, lane, row0, col0 + c0, rows_full && c0 + kChunk <= ncols, c, ld_c, r, ld_r,
                           M, N);
        if (has_b) tmem_wait(vb);
        const bool has_next = c0 + 2 * kChunk < ncols;
        if (has_next) tmem_ld32(taddr + (uint32_t)(c0 + 2 * kChunk), va);
        if (has_b)
          emit_block<C_BF16>(vb, stage_f, lane, row0, col0 + c0 + kChunk, rows_full && c0 + 2 * kChunk <= ncols, c,
                             ld_c, r, ld_r, M, N);
        if (has_next) tmem_wait(va);
      }
      // this warp's share of the accumulator has been read: release it
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(a));
    }
    if (lane == 0 && tma_chunk > 0) bulk_wait_all();  // the tensor stores have landed
  }
  __syncwarp();
  if constexpr (SPLIT) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // the partial sums of every rank are in place
    if (warp >= 2 && have_acc) {
      // rank q finishes rows [q 128 / splits, (q + 1) 128 / splits) of the
      // tile: each element is the sum of the ranks' partials in rank order
      // (the same order whichever rank adds them), read through distributed
      // shared memory a row segment of 4 columns per thread, coalesced
      int mb, nb;
      tile_coords(t_first, m_tiles, n_tiles, group_m, mb, nb);
      const int col0 = nb * BN;
      const int ncols = N - col0 < BN ? N - col0 : BN;
      const int r_lo = rank * kBM / splits, r_hi = (rank + 1) * kBM / splits;
      constexpr int kTPR = BN / 4;                   // threads per row
      constexpr int kRowsPer = (kEpiWarps * 32) / kTPR;
      const int e = threadIdx.x - 64;                // 0..127
      const int cq = (e % kTPR) * 4;
      if (splits <= 4) {
        const uint32_t part0 = base;  // the partial sums sit at the start of every rank's ring
        // kBatch row passes at a time, every rank's partials for them loaded
        // before any is added, so the distributed-shared-memory round trips
        // overlap; each element is still summed in rank order (measured: with 3
        // ranks 6.6 against 7.1 us on the decode in_proj; with 8 ranks the plain
        // row loop below is faster, 4.8 against 6.2 us on the decode x_proj)
        constexpr int kBatch = 4;
        constexpr int batch = kBatch;
#pragma unroll 1
        for (int rr0 = r_lo + e / kTPR; rr0 < r_hi; rr0 += batch * kRowsPer) {
          float4 acc[kBatch];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (q < splits) {
              const uint32_t pq = dsmem_map(part0, q);
              float4 x[kBatch];
#pragma unroll
              for (int bi = 0; bi < kBatch; ++bi) {
                const int rr = rr0 + bi * kRowsPer;
                x[bi] = (bi < batch && rr < r_hi && cq < ncols)
                            ? dsmem_ld4(pq + (uint32_t)((rr * (BN + 4) + cq) * 4))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int bi = 0; bi < kBatch; ++bi) {
                if (q == 0) {
                  acc[bi] = x[bi];
                } else {
                  acc[bi].x += x[bi].x;
                  acc[bi].y += x[bi].y;
                  acc[bi].z += x[bi].z;
                  acc[bi].w += x[bi].w;
                }
              }
            }
          }
#pragma unroll
          for (int bi = 0; bi < kBatch; ++bi) {
            const int rr = rr0 + bi * kRowsPer;
            const int row = mb * kBM + rr;
            if (bi >= batch || rr >= r_hi || row >= M || cq >= ncols) continue;
            const int col = col0 + cq;
            float xs[4] = {acc[bi].x, acc[bi].y, acc[bi].z, acc[bi].w};
            if (vec_ok && cq + 4 <= ncols) {
              if (r) {
                const float4 rv = *reinterpret_cast<const float4*>(r + (int64_t)row * ld_r + col);
                xs[0] += rv.x;
                xs[1] += rv.y;
                xs[2] += rv.z;
                xs[3] += rv.w;
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
              for (int j = 0; j < 4 && cq + j < ncols; ++j) {
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
      } else {
        const float* part0 = reinterpret_cast<const float*>(gbase);
#pragma unroll 1
        for (int rr = r_lo + e / kTPR; rr < r_hi; rr += kRowsPer) {
          const int row = mb * kBM + rr;
          if (row >= M || cq >= ncols) continue;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int q = 0; q < splits; ++q) {
            const float4 x =
                *reinterpret_cast<const float4*>(cluster.map_shared_rank(part0, q) + rr * (BN + 4) + cq);
            if (q == 0) {
              acc = x;
            } else {
              acc.x += x.x;
              acc.y += x.y;
              acc.z += x.z;
              acc.w += x.w;
            }
          }
          const int col = col0 + cq;
          float xs[4] = {acc.x, acc.y, acc.z, acc.w};
          if (vec_ok && cq + 4 <= ncols) {
            if (r) {
              const float4 rv = *reinterpret_cast<const float4*>(r + (int64_t)row * ld_r + col);
              xs[0] += rv.x;
              xs[1] += rv.y;
              xs[2] += rv.z;
              xs[3] += rv.w;
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
            for (int j = 0; j < 4 && cq + j < ncols; ++j) {
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
    }
    cluster.sync();  // every rank has read its peers' shared memory
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::kTmemCols) : "memory");
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

template <int BN, bool C_BF16, bool SPLIT>
cudaError_t launch_bn(const GemmArgs& g, const CUtensorMap& ma, const CUtensorMap& mw, int sms, int splits,
                      cudaStream_t stream) {
  auto kern = gemm_bf16_kernel<BN, C_BF16, SPLIT>;
  using Smem = GemmSmem<BN, SPLIT ? 3 : 8>;
  static int configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!__atomic_load_n(&configured[dev], __ATOMIC_RELAXED)) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::kAlloc)) !=
        cudaSuccess)
      return e;
    __atomic_store_n(&configured[dev], 1, __ATOMIC_RELAXED);
  }
  const int64_t tiles = ((g.M + kBM - 1) / kBM) * ((g.N + BN - 1) / BN);
  const uintptr_t cp = reinterpret_cast<uintptr_t>(g.c), rp = reinterpret_cast<uintptr_t>(g.r);
  const int vec_ok = (cp % (C_BF16 ? 8 : 16)) == 0 && g.ld_c % 4 == 0 && (!g.r || (rp % 16 == 0 && g.ld_r % 4 == 0));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(SPLIT ? tiles * splits : (tiles < sms ? tiles : sms)));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem::kAlloc;
  cfg.stream = stream;
  // programmatic dependent launch: this grid's set-up (barriers, tensor
  // memory) overlaps the previous kernel's tail; its first global access waits
  // for that kernel (griddepcontrol.wait)
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = SPLIT ? 2 : 1;
  // row blocks per group: their A rows take at most ~24 MB of L2 (measured on
  // the 2.8b in_proj and out_proj: 48 MB groups are evicted between the waves
  // of a group by the output stream, 16-row-block groups re-read the weight)
  const int64_t m_tiles = (g.M + kBM - 1) / kBM;
  int64_t group_m = (int64_t)24e6 / ((int64_t)kBM * g.K * 2);
  group_m = group_m < 8 ? 8 : (group_m > m_tiles ? m_tiles : group_m);
  // bf16 output without a residual goes out through tensor stores: C 16-byte
  // aligned with 16-byte rows
  CUtensorMap mc = ma;
  const int c_tma = C_BF16 && !SPLIT && !g.r && (cp % 16) == 0 && (g.ld_c * 2) % 16 == 0 &&
                    make_map(&mc, g.c, g.M, g.N, g.ld_c, 32);
  return cudaLaunchKernelEx(&cfg, kern, ma, mw, mc, g.c, g.ld_c, g.r, g.ld_r, (int)g.M, (int)g.N, (int)g.K, vec_ok,
                            SPLIT ? splits : 1, (int)(group_m < 1 ? 1 : group_m), c_tma);
}

template <bool C_BF16, bool SPLIT>
cudaError_t launch_typed(const GemmArgs& g, int bn, const CUtensorMap& ma, const CUtensorMap& mw, int sms, int splits,
                         cudaStream_t stream) {
  if (bn == 64) return launch_bn<64, C_BF16, SPLIT>(g, ma, mw, sms, splits, stream);
  if (bn == 128) return launch_bn<128, C_BF16, SPLIT>(g, ma, mw, sms, splits, stream);
  if (bn == 192) return launch_bn<192, C_BF16, SPLIT>(g, ma, mw, sms, splits, stream);
  return launch_bn<256, C_BF16, SPLIT>(g, ma, mw, sms, splits, stream);
}

}  // namespace

// Tile width: the candidate with the least estimated time, (waves of tiles) x
// (BN + 32) -- a tile costs about its width plus a fixed share (its A tile,
// the epilogue's start) -- so small problems take narrower tiles that fill
// more SMs and large ones the wide tiles that halve the shared-memory traffic
// per MMA.
int gemm_tile_n(int64_t M, int64_t N, int sms) {
  int best = 256;
  int64_t best_cost = INT64_MAX;
  for (int bn : {256, 192, 128, 64}) {
    if (bn > 64 && N <= bn / 2) continue;  // no wider than needed
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
    const int64_t cost = ((tiles + sms - 1) / sms) * (bn + 32);
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// K split: when the output has at most half an SM's worth of tiles and K has
// at least 4 stages, clusters of up to 8 CTAs share a tile (at least two K
// stages each, no more CTAs than SMs).  It depends on the shape only, so a
// shape always sums its K in the same order.
int gemm_k_splits(int64_t M, int64_t N, int64_t K, int bn, int sms) {
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
  const int64_t k_tiles = (K + kBK - 1) / kBK;
  if (tiles * 2 > sms || k_tiles < 4) return 1;
  int64_t sp = k_tiles / 2;
  if (sp > 8) sp = 8;
  if (sp > sms / tiles) sp = sms / tiles;
  return sp >= 2 ? (int)sp : 1;
}

cudaError_t launch_gemm_bf16(const GemmArgs& g, cudaStream_t stream) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int bn = gemm_tile_n(g.M, g.N, sms);
  const int splits = gemm_k_splits(g.M, g.N, g.K, bn, sms);
  CUtensorMap ma, mw;
  if (!make_map(&ma, g.a, g.M, g.K, g.ld_a, kBM) || !make_map(&mw, g.w, g.N, g.K, g.ld_w, bn))
    return cudaErrorInvalidValue;
  if (splits > 1)
    return g.c_bf16 ? launch_typed<true, true>(g, bn, ma, mw, sms, splits, stream)
                    : launch_typed<false, true>(g, bn, ma, mw, sms, splits, stream);
  return g.c_bf16 ? launch_typed<true, false>(g, bn, ma, mw, sms, 1, stream)
                  : launch_typed<false, false>(g, bn, ma, mw, sms, 1, stream);
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
