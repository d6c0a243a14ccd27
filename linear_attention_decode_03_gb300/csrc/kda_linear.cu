// kda_linear.cu -- the layer's projections around the KDA core on GB300
// (sm_103a): y[M, N] = x[M, K] . W[N, K]^T, bf16 in and out, fp32 accumulation
// (see include/kda.h, kda_linear).
//
// Sources: the K1 page ("vllm.models.kimi_k3.amd.specialized_decode.mono.
// attention.kda", module docstring) gives the layer's in_proj GEMV in front
// of the KDA core -- x [rows, 7168] to the packed projection row -- and the
// K2a page ("vllm.models.kimi_k3.amd.specialized_decode.mono.attention.back",
// module docstring: K2a attn_post) the o_proj GEMV after it (core_out [rows, D] to
// [rows, 7168]); both weights are [out_features, in_features], the layout of
// a torch Linear.
//
// At decode batch sizes the product is bound by streaming the weight from
// HBM once (90 MB for in_proj at 12 heads), not by the tensor pipe: 2 x rows
// flops per weight element.  A CTA owns NB output columns and streams their
// weight rows (and the matching x rows) through a shared-memory ring fed by
// TMA tensor copies (cp.async.bulk.tensor, 64 x rows boxes, 128-byte swizzle,
// completing on an mbarrier per slot), while its warps load fragments with
// ldmatrix and multiply with m16n8k16 bf16 tensor instructions, for up to 16
// rows: one 16-row tile, 32 columns, 4 warps (one 8-column n-tile each), K in
// stages of 128, six stages of 12 KB: the bytes are weight.  (The template
// also takes 64-row passes over 128-column tiles with 8 warps; more than 16
// rows go to the tcgen05 kernel below instead: at 64 rows it measured 30.8
// against 35.8 us, while at 1-8 rows this kernel is the faster one, 13.0
// against 15.0 us for the 2-head in_proj.)
// Rows past `rows`, weight rows past N and k past K are outside the tensor
// maps: the copy engine fills them with zeros.
//
// Column tiles alone give too few CTAs to keep HBM busy (37 for the 2-head
// in_proj on 152 SMs), so K is split over a thread-block cluster of C CTAs
// (C <= 8): each CTA streams 1/C of the K stages, leaves its fp32 partial
// tile in its own shared memory, and after a cluster barrier each CTA sums
// 1/C of the tile's elements over the C partials through distributed shared
// memory and writes them out -- no global scratch, no atomics, and the sum is
// taken in the same order (rank 0 first) for every element.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kda.h"
#include "internal.h"

namespace {

constexpr int LIN_MAX_SPLIT = 8;  // portable cluster size
constexpr int LIN_KMULT = 8;      // K must be a multiple of this (16-byte weight rows)
constexpr int LIN_BOXK = 64;      // k a TMA box (128 bytes: the swizzle span)
constexpr long long LIN_WAIT_LIMIT = 2000000000ll;  // SM cycles (~1 s) before a copy wait gives up

// Tile shape: MB rows a pass and NB columns a CTA; KS k a stage in KS / 64
// boxes; a stage holds the x boxes (MB rows x 128 bytes each), then the weight
// boxes (NB rows).  Warp w takes rows 16 (w % WM) .. + 15 against n-tiles
// NT (w / WM) .. + NT - 1.
template <int MB, int NB>
struct LinShape {
  static constexpr int WARPS = MB == 16 ? 4 : 8;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int KS = MB == 16 ? 128 : 64;
  static constexpr int STAGES = MB == 16 ? 6 : 4;
  static constexpr int NBOX = KS / LIN_BOXK;
  static constexpr int XBOX = MB * 128;  // bytes
  static constexpr int WBOX = NB * 128;  // bytes
  static constexpr int STAGE = NBOX * (XBOX + WBOX);
  static constexpr int WM = MB / 16;                  // warps along the rows
  static constexpr int NT = NB / 8 / (WARPS / WM);    // n-tiles a warp
  static constexpr int RED = THREADS * NT * 4;        // fp32 partials a CTA
  static constexpr int RING = STAGES * STAGE;
  static constexpr int SMEM = 1024 + RING + 8 * STAGES;  // + 1024-byte alignment slack + an mbarrier a slot
  static_assert(WARPS % WM == 0 && NT >= 1 && (NT == 1 || NT % 2 == 0), "warp tiling");
  static_assert(XBOX % 1024 == 0 && WBOX % 1024 == 0, "boxes start on the swizzle pattern's 1 KB period");
  static_assert(RED * 4 <= RING, "partials overlay the ring");
  static_assert(NB <= 256 && MB <= 256, "a TMA box is at most 256 rows");
};

// Sticky device-side error bits of the projections (KDA_ERR_TIMEOUT), read and
// cleared by kda_linear_check.
__device__ unsigned g_lin_err;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte address of 16-byte chunk `chunk` (0..7) of row `row` of a box written
// with the 128-byte swizzle: the chunk index is XORed with the row mod 8.
__device__ __forceinline__ uint32_t swz(uint32_t box, int row, int chunk) {
  return box + row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Phase `parity` of an mbarrier, or false after LIN_WAIT_LIMIT cycles.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long c0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - c0 > LIN_WAIT_LIMIT) return false;
  return true;
}
// One 2-D TMA box (coordinates: k, row) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap* map, int k, int row, uint32_t bar,
                                        unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(k), "r"(row), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

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
// 16 bytes at the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ float4 ld_peer_f32x4(const float* local, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote));
  return v;
}
// Sum of the `split` CTAs' four floats at `local` (CTA ranks q < split), in
// rank order; every load is issued before the first add, so the distributed-
// shared-memory round trips overlap.
__device__ __forceinline__ float4 cluster_sum4(const float* local, unsigned split) {
  float4 t[LIN_MAX_SPLIT];
#pragma unroll
  for (int q = 0; q < LIN_MAX_SPLIT; ++q)
    t[q] = (unsigned)q < split ? ld_peer_f32x4(local, q) : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 v = t[0];
#pragma unroll
  for (int q = 1; q < LIN_MAX_SPLIT; ++q) {
    v.x += t[q].x;
    v.y += t[q].y;
    v.z += t[q].z;
    v.w += t[q].w;
  }
  return v;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct LinArgs {
  __nv_bfloat16* y;
  long long ldy;
  long long M, N, K;
  unsigned x_box_bytes;  // bytes of one x box: its rows (min(rows, MB)) x 128
  int y_vec;             // y and ldy allow 16-byte stores (y 16-byte aligned, ldy % 8 == 0)
  int y_vec8;            // y and ldy allow 8-byte stores (y 8-byte aligned, ldy % 4 == 0)
};

// Issued by one thread: the weight boxes of stage k0 .. k0 + KS into ring slot
// `st`, with `bar` told to expect the whole stage (weight and x boxes).
template <int MB, int NB>
__device__ __forceinline__ void issue_stage_w(const LinArgs& a, const CUtensorMap* tmw, uint32_t st, uint32_t bar,
                                              long long n0, long long k0) {
  using T = LinShape<MB, NB>;
  unsigned long long w_policy;  // the weight is read once
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(w_policy));
  mbar_expect_tx(bar, T::NBOX * (a.x_box_bytes + T::WBOX));
#pragma unroll
  for (int b = 0; b < T::NBOX; ++b)
    tma_box(st + T::NBOX * T::XBOX + b * T::WBOX, tmw, (int)(k0 + b * LIN_BOXK), (int)n0, bar, w_policy);
}
// ... and its x boxes.
template <int MB, int NB>
__device__ __forceinline__ void issue_stage_x(const CUtensorMap* tmx, uint32_t st, uint32_t bar, long long m0,
                                              long long k0) {
  using T = LinShape<MB, NB>;
  unsigned long long x_policy;  // x is read by every CTA
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(x_policy));
#pragma unroll
  for (int b = 0; b < T::NBOX; ++b) tma_box(st + b * T::XBOX, tmx, (int)(k0 + b * LIN_BOXK), (int)m0, bar, x_policy);
}
// The x and weight boxes of stage k0 .. k0 + KS into ring slot `st`, all completing on `bar`.
template <int MB, int NB>
__device__ __forceinline__ void issue_stage(const LinArgs& a, const CUtensorMap* tmx, const CUtensorMap* tmw,
                                            uint32_t st, uint32_t bar, long long m0, long long n0, long long k0) {
  issue_stage_w<MB, NB>(a, tmw, st, bar, n0, k0);
  issue_stage_x<MB, NB>(tmx, st, bar, m0, k0);
}

template <int MB, int NB>
__global__ void __launch_bounds__(LinShape<MB, NB>::THREADS) kda_linear_kernel(
    const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw, const LinArgs a) {
  using T = LinShape<MB, NB>;
  constexpr int NT = T::NT, STAGES = T::STAGES;
  extern __shared__ __align__(128) unsigned char lsmem[];
  // the ring starts on a 1 KB boundary (the swizzle pattern's period)
  const uint32_t raw = smem_addr(lsmem);
  const uint32_t ring_s = (raw + 1023u) & ~1023u, bar0 = ring_s + T::RING;
  float* red = reinterpret_cast<float*>(lsmem + (ring_s - raw));  // the partial tile, over the drained ring
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wrow = (warp % T::WM) * 16, wnt = (warp / T::WM) * NT;  // the warp's rows and first n-tile
  // without a cluster launch each CTA is a cluster of one: rank 0 of 1
  const unsigned split = cluster_nctarank(), rank = cluster_ctarank();
  const long long n0 = (long long)cluster_id_x() * NB;
  const long long total = (a.K + T::KS - 1) / T::KS;  // k stages over the whole K (the last one zero-padded)
  const long long s_begin = total * rank / split;
  const long long stages = total * (rank + 1) / split - s_begin;
  // ldmatrix row addresses: lane l feeds row l & 7 of 8x8 matrix l >> 3
  const int lr = lane & 7, lm = lane >> 3;

  // the first pass's prologue stages, whose weight boxes go out at once: they depend
  // on no earlier kernel (the x boxes follow after the dependent-launch wait)
  const long long early = stages < STAGES - 1 ? stages : STAGES - 1;
  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
    for (int i = 0; i < STAGES; ++i) mbar_init(bar0 + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (long long s = 0; s < early; ++s)
      issue_stage_w<MB, NB>(a, &tmw, ring_s + (uint32_t)s * T::STAGE, bar0 + 8 * (uint32_t)s, n0,
                            (s_begin + s) * T::KS);
  }
  __syncthreads();

  // As a programmatic dependent (a layer plan's o_proj) the set-up above and the
  // first weight boxes overlap the previous kernel's tail; x is its output.
  // Otherwise a no-op.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  bool dead = false;  // a copy wait gave up: no more copies, outputs not meaningful
  long long g0 = 0;   // ring stages used by earlier passes (slot and phase bookkeeping)
  for (long long m0 = 0; m0 < a.M; m0 += MB, g0 += stages) {
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    const long long run = dead ? 0 : stages;
    if (threadIdx.x == 0) {  // ring prologue: stages 0 .. STAGES-2 in flight
      for (int s = 0; s < STAGES - 1 && s < run; ++s) {
        const uint32_t slot = (uint32_t)((g0 + s) % STAGES);
        if (g0 == 0 && s < early)  // the first pass: its weight boxes are already out
          issue_stage_x<MB, NB>(&tmx, ring_s + slot * T::STAGE, bar0 + 8 * slot, m0, (s_begin + s) * T::KS);
        else
          issue_stage<MB, NB>(a, &tmx, &tmw, ring_s + slot * T::STAGE, bar0 + 8 * slot, m0, n0,
                              (s_begin + s) * T::KS);
      }
    }
    long long issued = run < STAGES - 1 ? run : STAGES - 1;
    for (long long s = 0; s < run; ++s) {
      const long long g = g0 + s;
      const uint32_t slot = (uint32_t)(g % STAGES);
      const bool ok = mbar_wait_bounded(bar0 + 8 * slot, (unsigned)((g / STAGES) & 1));
      // every warp is past stage s-1 (its slot is free again) and agrees on the outcome
      if (__syncthreads_or(!ok)) {
        dead = true;
        if (threadIdx.x == 0) atomicOr(&g_lin_err, KDA_ERR_TIMEOUT);
        for (long long q = s; q < issued; ++q)  // the copies still in flight land before the CTA moves on
          mbar_wait_bounded(bar0 + 8 * (uint32_t)((g0 + q) % STAGES), (unsigned)(((g0 + q) / STAGES) & 1));
        break;
      }
      const long long next = s + STAGES - 1;
      if (next < run) {
        if (threadIdx.x == 0) {
          const uint32_t ns = (uint32_t)((g0 + next) % STAGES);
          issue_stage<MB, NB>(a, &tmx, &tmw, ring_s + ns * T::STAGE, bar0 + 8 * ns, m0, n0,
                              (s_begin + next) * T::KS);
        }
        issued = next + 1;
      }
      const uint32_t xs = ring_s + slot * T::STAGE, ws = xs + T::NBOX * T::XBOX;
      if (NT == 1) {
        // one n-tile: B fragments of two k16 steps in one ldmatrix.x4
#pragma unroll
        for (int kk = 0; kk < T::KS / 16; kk += 2) {
          const int box = kk >> 2, c0 = 2 * (kk & 3);
          uint32_t a0[4], a1[4], b[4];
          ldsm_x4(a0, swz(xs + box * T::XBOX, wrow + lr + (lm & 1) * 8, c0 + (lm >> 1)));
          ldsm_x4(a1, swz(xs + box * T::XBOX, wrow + lr + (lm & 1) * 8, c0 + 2 + (lm >> 1)));
          ldsm_x4(b, swz(ws + box * T::WBOX, wnt * 8 + lr, c0 + lm));
          mma_bf16(acc[0], a0[0], a0[1], a0[2], a0[3], b[0], b[1]);
          mma_bf16(acc[0], a1[0], a1[1], a1[2], a1[3], b[2], b[3]);
        }
      } else {
        // the warp's 16 rows against its NT n-tiles, two n-tiles an ldmatrix.x4
#pragma unroll
        for (int kk = 0; kk < T::KS / 16; ++kk) {
          const int box = kk >> 2, c0 = 2 * (kk & 3);
          const uint32_t xb = xs + box * T::XBOX, wb = ws + box * T::WBOX;
          uint32_t af[4];
          ldsm_x4(af, swz(xb, wrow + lr + (lm & 1) * 8, c0 + (lm >> 1)));
#pragma unroll
          for (int jp = 0; jp < NT / 2; ++jp) {
            uint32_t b[4];
            ldsm_x4(b, swz(wb, (wnt + 2 * jp + (lm >> 1)) * 8 + lr, c0 + (lm & 1)));
            mma_bf16(acc[2 * jp], af[0], af[1], af[2], af[3], b[0], b[1]);
            mma_bf16(acc[2 * jp + 1], af[0], af[1], af[2], af[3], b[2], b[3]);
          }
        }
      }
    }
    __syncthreads();  // every warp is done with the ring: the partials overlay it
    if (m0 + MB >= a.M) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // partial element e = ((j * 4 + c) * THREADS + thread): fragment c of the thread's n-tile j
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[(j * 4 + c) * T::THREADS + threadIdx.x] = acc[j][c];
    // these generic-proxy writes precede the next pass's tensor copies into the same bytes
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (split > 1) cluster_sync(); else __syncthreads();
    // this CTA's share of the tile: quads of elements [rank * Q / split, (rank + 1) * Q / split), Q = RED / 4
    constexpr int Q = T::RED / 4;
    const int q_end = (int)(Q * (rank + 1) / split);
    for (int qd = (int)(Q * rank / split) + threadIdx.x; qd < q_end; qd += T::THREADS) {
      const float4 v4 = split > 1 ? cluster_sum4(red + 4 * qd, split) : *reinterpret_cast<const float4*>(red + 4 * qd);
      const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // accumulator layout of m16n8: c0, c1 at row lane/4, columns 2 (lane % 4) + {0, 1}; c2, c3 eight rows down
        const int e = 4 * qd + i;
        const int t = e % T::THREADS, jc = e / T::THREADS, j = jc >> 2, c = jc & 3;
        const int tw = t >> 5, tl = t & 31;
        const long long m = m0 + (tw % T::WM) * 16 + (tl >> 2) + (c >> 1) * 8;
        const long long n = n0 + ((tw / T::WM) * NT + j) * 8 + (tl & 3) * 2 + (c & 1);
        if (m < a.M && n < a.N) a.y[m * a.ldy + n] = __float2bfloat16_rn(vv[i]);
      }
    }
    // the peers have read this CTA's partials before it refills the ring or exits
    if (split > 1) cluster_sync(); else __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// rows > 16: tcgen05 (5th-generation tensor core) tiles.  A CTA owns a
// 128 x 256 output tile, or 256 x 256 as two 128-row halves (rows past `rows`
// are the copy engine's zeros), K in stages of 64 through a ring of x boxes
// (16 KB a half) and a weight box (32 KB), all 128-byte swizzled: the
// canonical K-major layout of the MMA's shared-memory descriptors.  Warp 0's
// lane 0 issues the TMA copies, warp 1's lane 0 the MMAs (M 128, N 256, K 16;
// four a stage and half) into a 256-column fp32 accumulator a half in tensor
// memory; each stage's commit frees its ring slot.  After the last stage the
// four warps read the accumulators (warp w: lanes = rows 32w .. 32w + 31) and
// write bf16 rows, or, with K split over a cluster as in the kernel above, put
// the fp32 partial tile in shared memory (row-major, padded) and sum it over the
// cluster through distributed shared memory.  Few rows make the weight the
// bytes (x : W = 1 : 2 a stage); with many rows the bytes each SM takes in per
// product bound the tiles as much as the tensor pipe does, which the two-half
// tile cuts by a third (see TcShape).  Every CTA loads its own boxes: the copies
// only ever read this GPU's memory through the caller's tensor maps.
constexpr int TC_BM = 128, TC_BK = 64, TC_THREADS = 128;
constexpr int TC_ABYTES = TC_BM * 128;  // one 64-k x box
// MH row halves a CTA, BN weight rows (tile columns): MH = 1 a 128 x BN tile, MH = 2 a
// 256 x BN tile whose two 128-row halves share each weight box (two M128 MMAs a k
// step into two BN-column accumulators).  The two-half tile takes a third fewer
// bytes into the SM per product (64 KB a stage for 256 x 256 x 64 against 48 KB for
// 128 x 256 x 64), the intake that bounds these tiles with many rows; narrower
// tiles give more CTAs where the tiles are few.
template <int MH, int BN>
struct TcShape {
  static constexpr int BM = TC_BM * MH;
  static constexpr int BBYTES = BN * 128;  // one 64-k weight box
  static constexpr int STAGE = MH * TC_ABYTES + BBYTES;
  static constexpr int STAGES = (200 * 1024) / STAGE > 8 ? 8 : (200 * 1024) / STAGE;  // ring <= 200 KB
  static constexpr int RING = STAGES * STAGE;
  static constexpr int SMEM = 1024 + RING + 8 * (2 * STAGES + 1) + 16;
  // one fp32 accumulator of BN columns a half; the allocation a power of two >= 32
  static constexpr int TMEM_COLS = BN * MH <= 32    ? 32
                                   : BN * MH <= 64  ? 64
                                   : BN * MH <= 128 ? 128
                                   : BN * MH <= 256 ? 256
                                                    : 512;
  // partial tile, row-major: element (r, c) at r * RED_LD + c (16-byte stores, no bank conflicts)
  static constexpr int RED_LD = BN + 4;
  // tcgen05 instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
  // and B (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
  // M >> 4 at bits 24-28.
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                    ((uint32_t)(TC_BM >> 4) << 24);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "an M128 MMA takes N = 16..256 in steps of 16");
  static_assert(STAGE % 1024 == 0, "stages start on 1024-byte swizzle atoms");
  static_assert(STAGES >= 3, "at least three stages in flight");
  static_assert(TC_BM * RED_LD * 4 <= RING, "a half's partials overlay the ring");
  static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};
// Time model of these tiles, in microseconds, for picking MH, BN and the K split C
// (fitted to 45 measured in_proj / o_proj shapes -- 2, 12 and 96 heads, 17 to 1024
// rows, K 256 to 12288 -- at every MH, BN and C, each constant held to a
// physically plausible range): a CTA runs its S / C stages of 64 k at
//   s = max(MMA time (~ MH x BN), the SM's own intake time (~ the stage's bytes),
//           n x the share of the GPU's L2 intake a CTA takes (~ the stage's bytes))
// (n = CTAs running at once), plus a fixed part (first copies, accumulator
// read-out, stores; more for two halves, and growing with the tile's rows x
// columns), plus the split's partial-tile reduction (~ MH x BN) when C > 1; the
// kernel's time is that CTA time x the waves of clusters.
struct TcModel {
  double mma;        // us a stage of 128 x 256 x 64 products
  double sm_intake;  // us a 48 KB stage
  double l2_share;   // us a 48 KB stage per running CTA
  double fixed, fixed_two_halves, fixed_row;  // us; us more with MH = 2; us a tile row of 256 columns
  double reduce;     // us a 128 x 256 partial tile
};
constexpr TcModel TC_MODEL = {0.287, 0.413, 0.00306, 11.05, 5.05, 0.0233, 1.71};

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// whose 8-row x 128-byte swizzle atoms are stacked every 1024 bytes: start
// address >> 4 (bits 0-13), leading offset (bits 16-29; not used by this
// layout, set to 1), stride between atoms 1024 >> 4 (bits 32-45), the fixed
// 0b001 at bits 46-48, base offset 0 (the atoms start on 1024-byte
// boundaries), swizzle mode 2 (128-byte) at bits 61-63.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

template <int MH, int BN>
__global__ void __launch_bounds__(TC_THREADS, 1) kda_linear_tc_kernel(const __grid_constant__ CUtensorMap tmx,
                                                                    const __grid_constant__ CUtensorMap tmw,
                                                                    const LinArgs a, int tiles_m) {
  using T = TcShape<MH, BN>;
  constexpr int TC_STAGES = T::STAGES, TC_STAGE = T::STAGE, TC_RING = T::RING;
  extern __shared__ __align__(128) unsigned char tsmem[];
  const uint32_t raw = smem_addr(tsmem);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t full0 = ring + TC_RING, empty0 = full0 + 8 * TC_STAGES, accum_bar = empty0 + 8 * TC_STAGES;
  const uint32_t tmem_slot = accum_bar + 8;  // tcgen05.alloc writes the accumulator's address here
  unsigned char* ring_p = tsmem + (ring - raw);
  float* red = reinterpret_cast<float*>(ring_p);
  volatile uint32_t* tmem_slot_p = reinterpret_cast<volatile uint32_t*>(ring_p + (tmem_slot - ring));
  volatile int* consumed_p = reinterpret_cast<volatile int*>(ring_p + (tmem_slot - ring) + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // cluster = the split CTAs of one output tile: rank = K part
  const unsigned split = cluster_nctarank(), rank = cluster_ctarank();
  const long long grp = cluster_id_x();
  // the row tiles of one column tile are neighbours in launch order, so they run
  // together and all but the first find the weight boxes in L2
  const long long m0 = (grp % tiles_m) * T::BM, n0 = (grp / tiles_m) * BN;
  const long long total = (a.K + TC_BK - 1) / TC_BK;
  const long long s_begin = total * rank / split;
  const long long stages = total * (rank + 1) / split - s_begin;

  // Thread 0 is also the producer's issuing lane (warp 0, lane 0): its cache policies, and
  // the stages whose weight box it puts in flight at once.
  unsigned long long w_policy = 0, x_policy = 0;
  const long long early = stages < TC_STAGES ? stages : TC_STAGES;
  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
    for (int i = 0; i < TC_STAGES; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    mbar_init(accum_bar, 1);
    *consumed_p = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the weight tile is read once when there is one row tile (evict first), else kept for the others
    if (a.M <= T::BM)
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(w_policy));
    else
      asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(w_policy));
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(x_policy));
    // The weight boxes of the first stages depend on no earlier kernel: they go out
    // before the tensor memory, the barrier and (as a dependent launch) the wait for x.
    // Each stage's barrier expects the whole stage; its x boxes follow in the loop below.
    for (long long s0 = 0; s0 < early; ++s0) {
      const uint32_t bar = full0 + 8 * (uint32_t)s0;
      mbar_expect_tx(bar, TC_STAGE);
      tma_box(ring + (uint32_t)s0 * TC_STAGE + MH * TC_ABYTES, &tmw, (int)((s_begin + s0) * TC_BK), (int)n0, bar,
              w_policy);
    }
  }
  if (warp == 0) {  // the accumulators: 128 lanes x 256 fp32 columns of tensor memory a half
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                 "r"(T::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot_p;
  // As a programmatic dependent (a layer plan's o_proj) the set-up above and the
  // first weight boxes overlap the previous kernel's tail; x is its output.
  // Otherwise a no-op.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Warps 0 and 1 run their loops whole (converged, spinning on the barrier
  // without the sleep hint: a suspended thread wakes late), lane 0 issuing.
  bool ok_all = true;
  long long issued = 0;
  if (warp == 0) {  // producer (the first round's empty waits pass at once: every early stage gets its x)
    for (long long s = 0; s < stages; ++s) {
      const uint32_t slot = (uint32_t)(s % TC_STAGES);
      const bool ok = mbar_wait_bounded(empty0 + 8 * slot, (unsigned)(((s / TC_STAGES) & 1) ^ 1));
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        ok_all = false;
        break;
      }
      if (lane == 0) {
        const uint32_t st = ring + slot * TC_STAGE, bar = full0 + 8 * slot;
        const int k = (int)((s_begin + s) * TC_BK);
        if (s >= early) {  // the x box of each half and the weight box
          mbar_expect_tx(bar, TC_STAGE);
          tma_box(st + MH * TC_ABYTES, &tmw, k, (int)n0, bar, w_policy);
        }
#pragma unroll
        for (int hf = 0; hf < MH; ++hf) tma_box(st + hf * TC_ABYTES, &tmx, k, (int)(m0 + hf * TC_BM), bar, x_policy);
      }
      __syncwarp();
      issued = s + 1;
    }
  } else if (warp == 1) {  // MMA issuer
    long long s = 0;
    for (; s < stages; ++s) {
      const uint32_t slot = (uint32_t)(s % TC_STAGES);
      const bool ok = mbar_wait_bounded(full0 + 8 * slot, (unsigned)((s / TC_STAGES) & 1));
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        ok_all = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (lane == 0) {
        const uint32_t st = ring + slot * TC_STAGE;
#pragma unroll
        for (int k = 0; k < TC_BK / 16; ++k) {  // 16 k = 32 bytes along the swizzled row
          const uint64_t db = tc_desc(st + MH * TC_ABYTES + 32 * k);
          const uint32_t acc = (s > 0 || k > 0) ? 1u : 0u;
#pragma unroll
          for (int hf = 0; hf < MH; ++hf) {  // each half's rows against the shared weight box
            const uint64_t da = tc_desc(st + hf * TC_ABYTES + 32 * k);
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.u32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem + (uint32_t)(hf * BN)),
                "l"(da), "l"(db), "r"(T::IDESC), "r"(acc)
                : "memory");
          }
        }
        // the slot is free once these MMAs have read it
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(empty0 +
                                                                                                       8 * slot)
                     : "memory");
      }
      __syncwarp();
    }
    if (lane == 0) {
      *consumed_p = (int)s;
      // the accumulator is final once every MMA issued above has completed
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(accum_bar)
                   : "memory");
    }
    __syncwarp();
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // everyone: wait for the accumulator (no MMA at all when this CTA has no stages)
  bool have = stages > 0;
  if (have && !mbar_wait_bounded(accum_bar, 0)) ok_all = false;
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const bool dead = __syncthreads_or(!ok_all);
  if (threadIdx.x == 0 && dead) atomicOr(&g_lin_err, KDA_ERR_TIMEOUT);
  if (warp == 0 && lane == 0 && dead) {
    // copies issued but never consumed land before the ring is reused or the CTA exits
    for (long long q = *consumed_p; q < issued; ++q)
      mbar_wait_bounded(full0 + 8 * (uint32_t)(q % TC_STAGES), (unsigned)((q / TC_STAGES) & 1));
  }
  __syncthreads();
  const int r = warp * 32 + lane;
  // the rows of half hf of the tile that exist (0 past the end)
  auto rows_of = [&](int hf) {
    const long long left = a.M - (m0 + (long long)hf * TC_BM);
    return (int)(left <= 0 ? 0 : (left < TC_BM ? left : TC_BM));
  };
  // 32 accumulator columns c0.. of half hf for the warp's 32 lanes (rows)
  auto tmem_load = [&](int hf, int c0, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
          "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
          "=r"(v[30]), "=r"(v[31])
        : "r"(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(hf * BN + c0)));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  };
  if (split == 1) {
    // accumulator -> bf16 -> global: thread (warp w, lane l) owns row 32w + l of each half, 32 columns a load
#pragma unroll 1
    for (int hf = 0; hf < MH; ++hf) {
      const int rows_here = rows_of(hf);
      if (rows_here == 0) break;  // uniform across the CTA
      __nv_bfloat16* yr = a.y + (m0 + hf * TC_BM + r) * a.ldy;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        const int cw = BN - c0 < 32 ? BN - c0 : 32;  // columns of the tile in this load
        uint32_t v[32];
        if (have && !dead) {
          tmem_load(hf, c0, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
        if (r >= rows_here) continue;
        const long long n = n0 + c0;
        if (a.y_vec && n + cw <= a.N) {
          uint32_t p[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            p[j] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          uint4* dst = reinterpret_cast<uint4*>(yr + n);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (8 * q < cw) dst[q] = make_uint4(p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < cw && n + j < a.N) yr[n + j] = __float2bfloat16_rn(__uint_as_float(v[j]));
        }
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {  // the accumulators are read: give the tensor memory back
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T::TMEM_COLS) : "memory");
    }
    return;
  }
  // K split, one half at a time: accumulator -> shared memory (row-major, padded), 32
  // columns a load; rows past `rows` are not needed.  Every CTA of the cluster takes
  // part in both barriers of every half.
#pragma unroll 1
  for (int hf = 0; hf < MH; ++hf) {
    const int rows_here = rows_of(hf);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      const int cw = BN - c0 < 32 ? BN - c0 : 32;  // columns of the tile in this load
      uint32_t v[32];
      if (have && !dead && rows_here > 0) {
        tmem_load(hf, c0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
      if (r < rows_here) {
        float4* dst = reinterpret_cast<float4*>(red + r * T::RED_LD + c0);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (4 * q < cw)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync();
    if (hf == MH - 1 && warp == 0) {  // the accumulators are read: give the tensor memory back
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T::TMEM_COLS) : "memory");
    }
    // this CTA's share of the half: (row, 4-column group) pairs in row-major order, each
    // summed over the cluster's partials with 16-byte loads and stored as 4 bf16
    constexpr int CQ = BN / 4;
    const int E = rows_here * CQ;
    const int e_end = (int)((long long)E * (rank + 1) / split);
    for (int e = (int)((long long)E * rank / split) + threadIdx.x; e < e_end; e += TC_THREADS) {
      const int rr = e / CQ, cq = e % CQ;
      const float4 v4 = cluster_sum4(red + rr * T::RED_LD + 4 * cq, split);
      const long long n = n0 + 4 * cq;
      __nv_bfloat16* yr = a.y + (m0 + hf * TC_BM + rr) * a.ldy;
      if (a.y_vec8 && n + 4 <= a.N) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v4.x, v4.y), hi = __floats2bfloat162_rn(v4.z, v4.w);
        *reinterpret_cast<uint2*>(yr + n) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
      } else {
        const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (n + i < a.N) yr[n + i] = __float2bfloat16_rn(vv[i]);
      }
    }
    // the peers have read this CTA's partials before they are overwritten or it exits
    cluster_sync();
  }
}

bool lin_aligned(const void* p, unsigned n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// True when p is device memory of the current device: the tensor maps and the
// stores of these kernels address this GPU's own memory only.
bool on_current_device(const void* p) {
  int dev = 0;
  cudaPointerAttributes at;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear a lookup failure (an unknown host pointer) from the thread's error state
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (no link to libcuda).
EncodeTiled encode_fn() {
  static std::atomic<EncodeTiled> cached{nullptr};
  EncodeTiled fn = cached.load(std::memory_order_acquire);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiled>(p);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// A bf16 matrix [rows, cols] with row stride ld (elements) as 64 x box_rows boxes, 128-byte swizzle.
bool encode_map(CUtensorMap* map, const void* base, long long rows, long long cols, long long ld, int box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)LIN_BOXK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K split C (<= 8, <= the K stages): a CTA's time is about its share of the
// stages plus a fixed part (the first copies' latency, the reduction and the
// stores), so the kernel's is about waves x (stages / C + F), waves = the
// tiles over the clusters of C that the GPU holds at once
// (cudaOccupancyMaxActiveClusters -- a cluster must fit one GPC, so large
// clusters fit fewer times than the SM count suggests -- capped by the
// resident CTA slots), rounded up; the smallest C that minimises that.
constexpr double LIN_FIXED_STAGES = 4.0;  // F for the mma.sync tiles, in stages (measured per-stage ~0.5 us)
template <int MB, int NB>
int lin_launch(const void* x, long long ldx, const void* w, LinArgs a, cudaStream_t st, bool pdl) {
  using T = LinShape<MB, NB>;
  const long long tiles = (a.N + NB - 1) / NB;
  const int box_rows = (int)(a.M < MB ? a.M : MB);
  a.x_box_bytes = (unsigned)box_rows * 128u;
  CUtensorMap tmx, tmw;
  if (!encode_map(&tmx, x, a.M, a.K, ldx, box_rows) || !encode_map(&tmw, w, a.N, a.K, a.K, NB)) return KDA_ECUDA;
  // the shared-memory attribute is per device and cheap: set on every call
  if (cudaFuncSetAttribute(kda_linear_kernel<MB, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
      cudaSuccess)
    return KDA_ECUDA;
  // clusters of each size the device holds at once, looked up once per device and shape
  // looked up once per device (relaxed atomics: callers on several host threads
  // at worst repeat the same lookup)
  static std::atomic<int> cluster_cache[64][LIN_MAX_SPLIT + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(T::THREADS, 1, 1);
  cfg.dynamicSmemBytes = T::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the previous kernel ends
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const long long stages = (a.K + T::KS - 1) / T::KS;
  long long split = 1;
  double best = 1e300;
  for (int c = 1; c <= LIN_MAX_SPLIT && c <= stages; ++c) {
    int held = dev < 64 ? cluster_cache[dev][c].load(std::memory_order_relaxed) : 0;
    if (held <= 0) {
      attr[0].val.clusterDim.x = (unsigned)c;
      cfg.gridDim = dim3((unsigned)c, 1, 1);
      int sms = 0, per_sm = 0;
      if (cudaOccupancyMaxActiveClusters(&held, kda_linear_kernel<MB, NB>, &cfg) != cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_linear_kernel<MB, NB>, T::THREADS, T::SMEM) !=
              cudaSuccess)
        return KDA_ECUDA;
      // never more clusters than the resident CTA slots hold
      const int cap = sms * (per_sm > 0 ? per_sm : 1) / c;
      if (held > cap) held = cap;
      if (held <= 0) continue;
      if (dev < 64) cluster_cache[dev][c].store(held, std::memory_order_relaxed);
    }
    const double cost = (double)((tiles + held - 1) / held) * ((double)stages / c + LIN_FIXED_STAGES);
    if (cost < best * (1.0 - 1e-9)) best = cost, split = c;
  }
  if (tiles * split > 0x7fffffffLL) return KDA_EINVAL;
  cfg.gridDim = dim3((unsigned)(tiles * split), 1, 1);
  attr[0].val.clusterDim.x = (unsigned)split;
  cfg.numAttrs = pdl ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, kda_linear_kernel<MB, NB>, tmx, tmw, a) != cudaSuccess) return KDA_ECUDA;
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

// The launch of one tcgen05 tile shape (MH row halves, BN columns): the K split
// (cluster size) the time model picks and its modelled time (us).
struct TcPlan {
  int mh = 1, bn = 256;
  long long tiles_m = 0, groups = 0, split = 1;
  double cost = 1e300;
};

template <int MH, int BN>
int tc_plan(const LinArgs& a, TcPlan* plan) {
  using T = TcShape<MH, BN>;
  const long long tiles_m = (a.M + T::BM - 1) / T::BM, tiles_n = (a.N + BN - 1) / BN;
  const long long groups = tiles_m * tiles_n;  // output tiles: clusters of one K part
  if (cudaFuncSetAttribute(kda_linear_tc_kernel<MH, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
      cudaSuccess)
    return KDA_ECUDA;
  static std::atomic<int> cluster_cache[64][LIN_MAX_SPLIT + 1];  // by cluster size, as above (per tile shape)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(TC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = T::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const long long stages = (a.K + TC_BK - 1) / TC_BK;
  constexpr TcModel m = TC_MODEL;
  const double tile_rows = (double)(a.M < T::BM ? a.M : T::BM);
  constexpr double area = MH * BN / 256.0, bytes = T::STAGE / 49152.0;  // relative to 128 x 256 x 64, 48 KB
  const double fixed = m.fixed + (MH == 2 ? m.fixed_two_halves : 0.0) + m.fixed_row * tile_rows * (BN / 256.0);
  plan->mh = MH;
  plan->bn = BN;
  plan->tiles_m = tiles_m;
  plan->groups = groups;
  for (int c = 1; c <= LIN_MAX_SPLIT && c <= stages; ++c) {
    const int cs = c;  // cluster size
    int held = dev < 64 ? cluster_cache[dev][cs].load(std::memory_order_relaxed) : 0;
    if (held <= 0) {
      int sms = 0, per_sm = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_linear_tc_kernel<MH, BN>, TC_THREADS, T::SMEM) !=
              cudaSuccess)
        return KDA_ECUDA;
      attr[0].val.clusterDim.x = (unsigned)cs;
      cfg.gridDim = dim3((unsigned)cs, 1, 1);
      if (cudaOccupancyMaxActiveClusters(&held, kda_linear_tc_kernel<MH, BN>, &cfg) != cudaSuccess) return KDA_ECUDA;
      // never more clusters than the resident CTA slots hold
      const int cap = sms * (per_sm > 0 ? per_sm : 1) / cs;
      if (held > cap) held = cap;
      if (held <= 0) continue;
      if (dev < 64) cluster_cache[dev][cs].store(held, std::memory_order_relaxed);
    }
    // waves of clusters: a last wave at least half full counts by its share, a smaller
    // one as a whole wave
    const double w = (double)groups / held;
    const double whole = (double)((groups + held - 1) / held), tail = w - (whole - 1.0);
    const double waves = w <= 1.0 ? 1.0 : (tail >= 0.5 ? w : whole);
    const double running = (double)(groups < held ? groups : held) * c;
    double s = m.mma * area > m.sm_intake * bytes ? m.mma * area : m.sm_intake * bytes;
    if (running * m.l2_share * bytes > s) s = running * m.l2_share * bytes;
    const double cost = waves * ((double)stages / c * s + fixed + (c > 1 ? m.reduce * area : 0.0));
    if (cost < plan->cost * (1.0 - 1e-9)) plan->cost = cost, plan->split = c;
  }
  return KDA_OK;
}

template <int MH, int BN>
int tc_launch(const void* x, long long ldx, const void* w, LinArgs a, cudaStream_t st, bool pdl, const TcPlan& p) {
  CUtensorMap tmx, tmw;
  if (!encode_map(&tmx, x, a.M, a.K, ldx, TC_BM) || !encode_map(&tmw, w, a.N, a.K, a.K, BN)) return KDA_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(TC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = TcShape<MH, BN>::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the previous kernel ends
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (p.groups * p.split > 0x7fffffffLL) return KDA_EINVAL;
  cfg.gridDim = dim3((unsigned)(p.groups * p.split), 1, 1);
  if (cudaLaunchKernelEx(&cfg, kda_linear_tc_kernel<MH, BN>, tmx, tmw, a, (int)p.tiles_m) != cudaSuccess)
    return KDA_ECUDA;
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

int tc_dispatch(const void* x, long long ldx, const void* w, const LinArgs& a, cudaStream_t st, bool pdl,
                const TcPlan& p) {
  if (p.mh == 2) {
    if (p.bn == 192) return tc_launch<2, 192>(x, ldx, w, a, st, pdl, p);
    return tc_launch<2, 256>(x, ldx, w, a, st, pdl, p);
  }
  if (p.bn == 192) return tc_launch<1, 192>(x, ldx, w, a, st, pdl, p);
  if (p.bn == 128) return tc_launch<1, 128>(x, ldx, w, a, st, pdl, p);
  return tc_launch<1, 256>(x, ldx, w, a, st, pdl, p);
}

template <int MH, int BN>
int tc_consider(const LinArgs& a, TcPlan* best) {
  TcPlan p;
  const int rc = tc_plan<MH, BN>(a, &p);
  if (rc == KDA_OK && p.cost < best->cost) *best = p;
  return rc;
}

// The tcgen05 tiles: the shape and K split the time model rates fastest -- one or
// two 128-row halves (two halves cut the bytes a product but halve the tiles) of
// 256, 192 or (one half) 128 columns (narrower tiles give more CTAs where the tiles
// are few).  Two halves of 128 columns move the bytes of one half of 256 with a
// larger fixed part, and never measured faster, so they are not built.
int lin_launch_tc(const void* x, long long ldx, const void* w, LinArgs a, cudaStream_t st, bool pdl) {
  TcPlan best;
  int rc = KDA_OK;
  if ((rc = tc_consider<1, 256>(a, &best)) != KDA_OK || (rc = tc_consider<1, 192>(a, &best)) != KDA_OK ||
      (rc = tc_consider<1, 128>(a, &best)) != KDA_OK)
    return rc;
  if (a.M > TC_BM) {
    if ((rc = tc_consider<2, 256>(a, &best)) != KDA_OK || (rc = tc_consider<2, 192>(a, &best)) != KDA_OK) return rc;
  }
  return tc_dispatch(x, ldx, w, a, st, pdl, best);
}

}  // namespace

int kda_linear_enqueue(const void* x, long long rows, long long ldx, const void* w, long long N, long long K,
                       void* y, long long ldy, void* cuda_stream, bool pdl) {
  if (rows < 0 || N < 1 || K < LIN_KMULT || K % LIN_KMULT != 0) return KDA_EINVAL;
  if (rows == 0) return KDA_OK;
  if (!x || !w || !y || ldx < K || ldy < N) return KDA_EINVAL;
  // tensor maps: 16-byte aligned bases and row strides; coordinates fit 32 bits
  if (!lin_aligned(x, 16) || !lin_aligned(w, 16) || (ldx % 8) != 0 || !lin_aligned(y, 2)) return KDA_EINVAL;
  if (K > 0x7fffffffLL || N > 0x7fffffffLL || rows > 0x7fffffffLL) return KDA_EINVAL;
  if (!on_current_device(x) || !on_current_device(w) || !on_current_device(y)) return KDA_EINVAL;
  // rows <= 16: the one-tile mma.sync shape (the bytes are the weight);
  // beyond: tcgen05 tiles (at 64 rows they beat 64 x 128 mma.sync tiles,
  // 30.8 against 35.8 us for the 12-head in_proj, although half their x box
  // is the copy engine's zeros)
  LinArgs a;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.ldy = ldy;
  a.M = rows;
  a.N = N;
  a.K = K;
  a.x_box_bytes = 0;
  a.y_vec = lin_aligned(y, 16) && (ldy % 8) == 0;
  a.y_vec8 = lin_aligned(y, 8) && (ldy % 4) == 0;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (rows <= 16) return lin_launch<16, 32>(x, ldx, w, a, st, pdl);
  return lin_launch_tc(x, ldx, w, a, st, pdl);
}

extern "C" int kda_linear(const void* x, long long rows, long long ldx, const void* w, long long N, long long K,
                          void* y, long long ldy, void* cuda_stream) {
  return kda_linear_enqueue(x, rows, ldx, w, N, K, y, ldy, cuda_stream, false);
}

extern "C" int kda_linear_check(void* cuda_stream, unsigned* device_flags) {
  if (!device_flags) return KDA_EINVAL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) return KDA_ECUDA;
  unsigned v = 0;
  const unsigned zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_lin_err, sizeof(v)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_lin_err, &zero, sizeof(zero)) != cudaSuccess)
    return KDA_ECUDA;
  *device_flags = v;
  return KDA_OK;
}
