// kda_linear.cu -- the layer's projections around the KDA core on GB300
// (sm_103a): y[M, N] = x[M, K] . W[N, K]^T, bf16 in and out, fp32 accumulation
// (see include/kda.h, kda_linear).
//
// Sources: the K1 page ("vllm.models.kimi_k3.amd.specialized_decode.mono.
// attention.kda", module docstring) gives the layer's in_proj GEMV in front
// of the KDA core -- x [rows, 7168] to the packed projection row -- and the
// K2a page ("...attn_post") the o_proj GEMV after it (core_out [rows, D] to
// [rows, 7168]); both weights are [out_features, in_features], the layout of
// a torch Linear.
//
// At decode batch sizes (rows <= 64) the product is bound by streaming the
// weight from HBM once (90 MB for in_proj at 12 heads), not by the tensor
// pipe: 2 rows x 2 flops per weight byte.  So a CTA owns 32 output columns
// and streams their weight rows through a six-deep ring of 16-byte cp.async
// copies (with the matching x tile), while its four warps multiply from
// shared memory with m16n8k16 bf16 tensor instructions.  Two shapes: up to
// 16 rows, one 16-row tile, a warp per 8 columns and K in stages of 128 (the
// ring's bytes are nearly all weight); beyond, 64-row passes (a warp per 16
// rows, all 32 columns) with K in stages of 64.
//
// 32-column tiles alone give too few CTAs to keep HBM busy (37 for the
// 2-head in_proj, 197 at 12 heads on 152 SMs), so K is split over a thread-
// block cluster of C CTAs (C <= 8, chosen so that the grid fills the SMs'
// resident slots once): each CTA streams 1/C of the K stages, leaves its fp32
// partial tile in its own shared memory, and after a cluster barrier each CTA
// sums 1/C of the tile's elements over the C partials through distributed
// shared memory and writes them out -- no global scratch, no atomics, and the
// sum is taken in the same order (rank 0 first) for every element.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace {

constexpr int LIN_NB = 32;        // output columns a CTA
constexpr int LIN_STAGES = 5;     // ring depth (three CTAs fit an SM)
constexpr int LIN_MAX_SPLIT = 8;  // portable cluster size
constexpr int LIN_THREADS = 128;  // 4 warps
constexpr int LIN_KMULT = 64;     // K must be a multiple of this

// Tile shape: MB rows a pass, KS k a stage; rows padded by 8 bf16 in shared
// memory so that the fragment loads hit 32 distinct banks.
template <int MB>
struct LinShape {
  static constexpr int KS = MB == 16 ? 128 : 64;
  static constexpr int LD = KS + 8;
  static constexpr int STAGE_ELEMS = (MB + LIN_NB) * LD;
  static constexpr int SMEM = LIN_STAGES * STAGE_ELEMS * 2;  // bytes
  static constexpr int NT = MB == 16 ? 1 : 4;                 // n-tiles (of 8 columns) a warp
  static constexpr int RED = LIN_THREADS * NT * 4;            // fp32 partials a CTA
  static_assert(RED * 4 <= SMEM, "partials overlay the ring");
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy; src_bytes = 0 fills the destination with zeros (no read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, unsigned src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_nctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_id_x() {
  unsigned r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// All threads of all CTAs of the cluster; release/acquire order the shared-
// memory writes before it with the peers' reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// fp32 at the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ float ld_peer_f32(const float* local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

struct LinArgs {
  const __nv_bfloat16* x;
  long long ldx;
  const __nv_bfloat16* w;  // [N, K]
  __nv_bfloat16* y;
  long long ldy;
  long long M, N, K;
};

// Stage s of the ring: x rows [m0, m0 + MB) and weight rows [n0, n0 + 32) over
// k [k0, k0 + KS), zeros where the rows run past M or N (no read there).
template <int MB>
__device__ __forceinline__ void load_stage(const LinArgs& a, __nv_bfloat16* st, long long m0, long long n0,
                                           long long k0) {
  using T = LinShape<MB>;
  constexpr int CPR = T::KS / 8;  // 16-byte chunks a row
  __nv_bfloat16* xs = st;
  __nv_bfloat16* ws = st + MB * T::LD;
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < (MB * CPR) / LIN_THREADS; ++i) {
    const int c = tid + i * LIN_THREADS;
    const int r = c / CPR, kc = (c % CPR) * 8;
    const bool in = m0 + r < a.M;
    const __nv_bfloat16* src = in ? a.x + (m0 + r) * a.ldx + k0 + kc : a.x;
    cp_async16(xs + r * T::LD + kc, src, in ? 16u : 0u);
  }
#pragma unroll
  for (int i = 0; i < (LIN_NB * CPR) / LIN_THREADS; ++i) {
    const int c = tid + i * LIN_THREADS;
    const int r = c / CPR, kc = (c % CPR) * 8;
    const bool in = n0 + r < a.N;
    const __nv_bfloat16* src = in ? a.w + (n0 + r) * a.K + k0 + kc : a.w;
    cp_async16(ws + r * T::LD + kc, src, in ? 16u : 0u);
  }
}

template <int MB>
__global__ void __launch_bounds__(LIN_THREADS) kda_linear_kernel(const LinArgs a) {
  using T = LinShape<MB>;
  constexpr int NT = T::NT;
  extern __shared__ __align__(128) unsigned char lsmem[];
  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(lsmem);
  float* red = reinterpret_cast<float*>(lsmem);  // the partial tile, over the drained ring
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  // without a cluster launch each CTA is a cluster of one: rank 0 of 1
  const unsigned split = cluster_nctarank(), rank = cluster_ctarank();
  const long long n0 = (long long)cluster_id_x() * LIN_NB;
  const long long total = a.K / T::KS;  // k stages over the whole K
  const long long s_begin = total * rank / split;
  const long long stages = total * (rank + 1) / split - s_begin;
  // the warp's 16 rows (within the pass) and first n-tile
  const int wrow = MB == 16 ? 0 : warp * 16;
  const int wnt = MB == 16 ? warp : 0;

  for (long long m0 = 0; m0 < a.M; m0 += MB) {
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    // ring prologue: stages 0 .. STAGES-2 in flight
#pragma unroll
    for (int s = 0; s < LIN_STAGES - 1; ++s) {
      if (s < stages) load_stage<MB>(a, ring + s * T::STAGE_ELEMS, m0, n0, (s_begin + s) * T::KS);
      cp_async_commit();
    }
    for (long long s = 0; s < stages; ++s) {
      cp_async_wait<LIN_STAGES - 2>();  // stage s has landed (this thread's copies) ...
      __syncthreads();                  // ... and everyone's; stage s-1's slot is free again
      const long long next = s + LIN_STAGES - 1;
      if (next < stages)
        load_stage<MB>(a, ring + (next % LIN_STAGES) * T::STAGE_ELEMS, m0, n0, (s_begin + next) * T::KS);
      cp_async_commit();
      const __nv_bfloat16* xs = ring + (s % LIN_STAGES) * T::STAGE_ELEMS;
      const __nv_bfloat16* ws = xs + MB * T::LD;
      const int r0 = wrow + gid;
#pragma unroll
      for (int kk = 0; kk < T::KS / 16; ++kk) {
        const int kb = kk * 16 + tig * 2;
        uint32_t af[4];
        af[0] = *reinterpret_cast<const uint32_t*>(xs + r0 * T::LD + kb);
        af[1] = *reinterpret_cast<const uint32_t*>(xs + (r0 + 8) * T::LD + kb);
        af[2] = *reinterpret_cast<const uint32_t*>(xs + r0 * T::LD + kb + 8);
        af[3] = *reinterpret_cast<const uint32_t*>(xs + (r0 + 8) * T::LD + kb + 8);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int nr = (wnt + j) * 8 + gid;
          uint32_t bf[2];
          bf[0] = *reinterpret_cast<const uint32_t*>(ws + nr * T::LD + kb);
          bf[1] = *reinterpret_cast<const uint32_t*>(ws + nr * T::LD + kb + 8);
          mma_bf16(acc[j], af, bf);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with the ring: the partials overlay it
    // partial element e = ((j * 4 + c) * 128 + thread): fragment c of n-tile j of a thread
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[(j * 4 + c) * LIN_THREADS + threadIdx.x] = acc[j][c];
    if (split > 1) cluster_sync(); else __syncthreads();
    // this CTA's share of the tile: elements [rank * RED / split, (rank + 1) * RED / split)
    const int e_end = (int)(T::RED * (rank + 1) / split);
    for (int e = (int)(T::RED * rank / split) + threadIdx.x; e < e_end; e += LIN_THREADS) {
      float v = 0.0f;
      for (unsigned q = 0; q < split; ++q) v += split > 1 ? ld_peer_f32(red + e, q) : red[e];
      const int t = e % LIN_THREADS, jc = e / LIN_THREADS, j = jc >> 2, c = jc & 3;
      const int tw = t >> 5, tl = t & 31;
      const long long m = m0 + (MB == 16 ? 0 : tw * 16) + (tl >> 2) + (c >> 1) * 8;
      const long long n = n0 + ((MB == 16 ? tw : 0) + j) * 8 + (tl & 3) * 2 + (c & 1);
      if (m < a.M && n < a.N) a.y[m * a.ldy + n] = __float2bfloat16_rn(v);
    }
    // the peers have read this CTA's partials before it refills the ring or exits
    if (split > 1) cluster_sync(); else __syncthreads();
  }
}

bool lin_aligned(const void* p, unsigned n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// K split: the largest C <= 8 (and <= the K stages) with tiles x C within the
// GPU's resident CTA slots, so that one wave covers the grid.
template <int MB>
int lin_launch(const LinArgs& a, long long tiles, cudaStream_t st) {
  using T = LinShape<MB>;
  // the shared-memory attribute is per device and cheap: set on every call
  if (cudaFuncSetAttribute(kda_linear_kernel<MB>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
      cudaSuccess)
    return KDA_ECUDA;
  // resident CTA slots of the device, looked up once per device and shape
  static long long slot_cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ECUDA;
  long long slots = dev < 64 ? slot_cache[dev] : 0;
  if (slots <= 0) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_linear_kernel<MB>, LIN_THREADS, T::SMEM) !=
            cudaSuccess)
      return KDA_ECUDA;
    slots = (long long)sms * (per_sm > 0 ? per_sm : 1);
    if (dev < 64) slot_cache[dev] = slots;
  }
  long long split = slots / tiles;
  if (split > LIN_MAX_SPLIT) split = LIN_MAX_SPLIT;
  if (split > a.K / T::KS) split = a.K / T::KS;
  if (split < 1) split = 1;
  if (tiles * split > 0x7fffffffLL) return KDA_EINVAL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * split), 1, 1);
  cfg.blockDim = dim3(LIN_THREADS, 1, 1);
  cfg.dynamicSmemBytes = T::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kda_linear_kernel<MB>, a) != cudaSuccess) return KDA_ECUDA;
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

}  // namespace

extern "C" int kda_linear(const void* x, long long rows, long long ldx, const void* w, long long N, long long K,
                          void* y, long long ldy, void* cuda_stream) {
  if (rows < 0 || N < 1 || K < LIN_KMULT || K % LIN_KMULT != 0) return KDA_EINVAL;
  if (rows == 0) return KDA_OK;
  if (!x || !w || !y || ldx < K || ldy < N) return KDA_EINVAL;
  // 16-byte copies: x and weight rows start on 16-byte boundaries
  if (!lin_aligned(x, 16) || !lin_aligned(w, 16) || (ldx % 8) != 0 || !lin_aligned(y, 2)) return KDA_EINVAL;
  const long long ctas = (N + LIN_NB - 1) / LIN_NB;
  if (ctas > 0x7fffffffLL) return KDA_EINVAL;
  // rows <= 16 (and K a multiple of its 128-k stage): the one-tile shape
  const bool small = rows <= 16 && K % LinShape<16>::KS == 0;
  LinArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.ldx = ldx;
  a.w = static_cast<const __nv_bfloat16*>(w);
  a.y = static_cast<__nv_bfloat16*>(y);
  a.ldy = ldy;
  a.M = rows;
  a.N = N;
  a.K = K;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  return small ? lin_launch<16>(a, ctas, st) : lin_launch<64>(a, ctas, st);
}
