// kda_step.cu -- GB300 (sm_103a) kernels and C ABI of the KDA decode /
// spec-verify core (see include/kda.h for the contract).
//
// Sources: the vLLM documentation pages
//   "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.kda" (K1
//   kda_pre module docstring: kda_stage, kda_conv, kda_gates, kda_recur,
//   kda_norm) and
//   "vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.kda.prepared"
//   (PreparedKda.__init__, _operands, run, decode_conv_weight).
//
// Design: one CTA of 8 warps per (request, head), up to three resident per
// SM, every global access issued as early as its address is known, so that a
// CTA spends two memory round trips before its compute:
//   * round trip 1 (issued at entry, by every thread, with no dependence):
//       the request's slots / accepted, the lane's share of the head's f_b
//       (4 rows x 16 k, two 16-byte loads a row), the f_a, out-gate and beta
//       values, the packed conv taps and bias of the thread's channels, and
//       for decode the conv input from the projected row.
//   * round trip 2 (once the slots are in): every thread validates them and
//       loads the rest of the conv inputs of its channels (the start window;
//       verify: and the projected x); thread 0 puts the 64 KiB start state of
//       (slot, head) in flight as four 16 KiB bulk async copies
//       (cp.async.bulk, L2 evict-first) on four mbarriers -- decode at once,
//       verify once its own conv inputs are in.
//   * while the state lands: the causal conv of the q, k, v channels over the
//       L tokens; z = f_b . f_a (4 channels x 16 k a lane with mixed-precision
//       bf16 FMAs, a reduce-scatter over 8 lanes, a closed-form bound on the
//       fp32 error), the lower-bound gate and e^g; the l2norm of q and k and
//       k^.q^ (warp t on token t); then the windows after each token go to
//       slots[r, t].
//   * recurrence: two passes over pairs of 32-row quarters of the state
//       (rows = v; each pass waits on its two copies); 16 lanes own a v row,
//       8 k values a lane, four rows a thread in registers across the L
//       tokens; S'^T k^ and S'^T q^ are reduced with one 16-lane
//       reduce-scatter; every token's new rows leave straight from registers
//       for slots[r, t] (decode: slots[b]) as streaming stores, 128-bit for
//       fp32 and 64-bit for bf16 (a shared-memory write-back and bulk store
//       needed a barrier a pass and measured no faster).
//   * gated RMSNorm, warp t on token t -> bf16 core_out.
// As an option (kda_set_v_split) a (request, head) runs as a cluster of two
// CTAs, each with 64 of the v rows (one recurrence pass) and half the outputs,
// the halves of o swapped through distributed shared memory for the norm.
// Decode of two rows or more runs rows 2p and 2p + 1 of one head in one CTA
// (kda_decode_pair_kernel): the rows share the load round trips and the head's
// f_b; two bf16 states sit side by side in the shared memory one fp32 state
// takes, and with an fp32 pool the second row's halves follow the first row's
// passes into the one state buffer.
// The bf16 hand-offs (conv outputs, z) are rounded correctly: each fp32 value
// carries a bound on its error and is recomputed exactly (fp64, or a
// compensated TwoSum sum) when the bound straddles a bf16 rounding boundary.
// Every wait is bounded (about 1 s of SM clock cycles); a wait that gives up
// sets KDA_ERR_TIMEOUT (see include/kda.h for what is then written).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"
#include "internal.h"

namespace {

constexpr int HD = 128;                        // head dim (k and v)
constexpr int THREADS = 256;                   // 8 warps
constexpr int WARPS = THREADS / 32;
constexpr int Z_CHANNELS = HD / WARPS;         // 16 decay channels a warp
constexpr int STATE_FLOATS = HD * HD;          // elements of one (slot, head) state
constexpr int QUARTERS = 4;
constexpr long long WAIT_LIMIT_CYCLES = 2000000000ll;  // ~1 s at 2 GHz

enum { TASK_OK = 0, TASK_PADDING = 1, TASK_SKIP = 2 };

struct StepArgs {
  const __nv_bfloat16* projected;
  long long pitch;
  __nv_bfloat16* conv_state;
  void* state_pool;             // fp32 or bf16 [pool, H, 128 (v), 128 (k)]
  long long pool;
  const int* slots;
  const int* accepted;
  __nv_bfloat16* out;
  const uint2* conv_w;          // prepared [3D]: the W taps right-aligned in 4, two bf16 a word
  const __nv_bfloat16* bias;    // [3D] or null
  const __nv_bfloat16* f_b;     // [D][128]
  const float* fb_norm;         // [D] Euclidean norm of each f_b row, rounded up
  const float* A_log;           // [H]
  const float* dt_bias;         // [D]
  const float* o_norm;          // [128]
  unsigned* err;
  float lb, eps, q_scale;
  int heads, D, W, conv_dim_first;
  int gate_mode;  // KDA_GATE_SIGMOID or KDA_GATE_SOFTPLUS
};

// Sizes of one (slot, head) state in the pool's storage type: fp32, or bf16
// (BS) when the handle's state pool holds bf16.
template <bool BS>
struct StateT {
  static constexpr int ELEM = BS ? 2 : 4;               // bytes an element
  static constexpr int BYTES = STATE_FLOATS * ELEM;     // 64 or 32 KiB
  static constexpr int QBYTES = BYTES / QUARTERS;       // one 32-row quarter
};

// Shared-memory carve-up for L tokens (byte offsets from the dynamic base).
template <int L, bool BS = false>
struct Smem {
  static constexpr int state = 0;                     // [128][128]        start state (storage type)
  static constexpr int eg = state + StateT<BS>::BYTES;  // float [L][128]  e^g
  static constexpr int kh = eg + L * HD * 4;          // float [L][128]    k, then k^
  static constexpr int qh = kh + L * HD * 4;          // float [L][128]    q, then q^
  static constexpr int fa = qh + L * HD * 4;          // bf16  [L][128]    f_a; later o
  static constexpr int vv = fa + L * HD * 2;          // bf16  [L][128]    v
  static constexpr int gate = vv + L * HD * 2;        // fp16  [L][128]    sigmoid(out-gate)
  static constexpr int fnp = gate + L * HD * 2;       // float [L][4]      partial sums of f_a^2
  static constexpr int beta = fnp + 16 * L;           // float [L]
  static constexpr int kq = beta + 4 * L;             // float [L]         k^.q^
  static constexpr int slot = kq + 4 * L;             // int   [L]         slots[r, t]
  static constexpr int ctl = slot + 4 * L;            // int   [2]         timeout flag
  static constexpr int mbar = (ctl + 8 + 7) / 8 * 8;  // u64   [4]
  static constexpr int bytes = mbar + 8 * QUARTERS;
};

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float bf_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
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

// As mbar_try_wait, but the thread may sleep up to SUSPEND_HINT_NS until the
// phase completes, instead of returning at once: a waiting warp then takes no
// issue slots from the warps that do the work it waits for.
constexpr unsigned SUSPEND_HINT_NS = 1000000u;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(SUSPEND_HINT_NS)
      : "memory");
  return ok != 0;
}

// Bulk async global -> shared copy completing on an mbarrier, L2 evict-first.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, unsigned bytes, uint32_t bar) {
  unsigned long long policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}


__device__ __forceinline__ void store_streaming_u2(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
// Two floats -> bf16x2 (nearest even), lo in the low half.
__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const unsigned*>(&v);
}

__device__ __forceinline__ void store_streaming(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// Packed fp32 pair arithmetic (two lanes of work per instruction on sm_100+),
// with the operands passed as plain registers.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// Sigmoid from the fast intrinsics: __expf is within 2 + 1.173 |x| ulp and
// __fdividef within 2 ulp (CUDA's documented bounds), so with the rounding of
// 1 + e^-x the result is within 2.35 |x| u + 2^-21 + u relative (u = 2^-24).
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// softplus(x) = log(1 + e^x) = max(x, 0) + log(1 + e^-|x|), fast intrinsics.
__device__ __forceinline__ float softplus_fast(float x) { return fmaxf(x, 0.0f) + __logf(1.0f + __expf(-fabsf(x))); }

// sqrt(s) for s >= 0 within 2^-21 relative (rsqrtf is within 2 ulp).
__device__ __forceinline__ float sqrt_fast(float s) { return s > 0.0f ? s * rsqrtf(s) : 0.0f; }

// ---- correctly rounded bf16 hand-offs ------------------------------------
// The conv outputs (q, k, v) and z = f_b . f_a are handed on as bf16.  They
// are computed in fp32 with a running bound on the fp32 error; when the fp32
// value lies within that bound of a bf16 rounding boundary, it is recomputed
// exactly enough (fp64, or a compensated fp32 sum) before rounding, so the
// bf16 value equals the correctly rounded one.
constexpr float U32 = 5.9604644775390625e-08f;  // 2^-24, fp32 unit roundoff

// True when rounding v to bf16 may differ from rounding a value within `bound` of v.
__device__ __forceinline__ bool bf16_rounding_uncertain(float v, float bound) {
  const unsigned a = __float_as_uint(v) & 0x7fffffffu;
  const float lo = __uint_as_float(a & 0xffff0000u);             // v truncated to bf16
  const float mid = __uint_as_float((a & 0xffff0000u) | 0x8000u); // lo + half a bf16 ulp
  return fabsf(__uint_as_float(a) - mid) <= bound || 2.0f * bound >= (mid - lo);
}

// fp64 -> bf16, round to nearest even, via round-to-odd to fp32 (fp32 keeps
// 16 more bits than bf16, so the second rounding is exact; Boldo & Melquiond,
// "Emulation of FMA and correctly rounded sums: proved algorithms using
// rounding to odd").
__device__ __forceinline__ float bf16_round_f64(double x) {
  const float f = __double2float_rz(x);
  unsigned b = __float_as_uint(f);
  if ((double)f != x) b |= 1u;
  return __bfloat162float(__float2bfloat16_rn(__uint_as_float(b)));
}

// bf16 (ties to even) of hi + lo, an unevaluated fp32 pair.  TwoSum first
// makes it s + e with s = fl(hi + lo) and |e| <= ulp(s) / 2.  Then s and s + e
// round alike unless s is itself a bf16 midpoint: any other fp32 value is at
// least one fp32 ulp from every midpoint, which e cannot cross.  At a midpoint
// the sign of e picks the neighbour, and e = 0 leaves the tie to even.
__device__ __forceinline__ float bf16_round_pair(float hi, float lo) {
  const float s = hi + lo, bp = s - hi;
  const float e = (hi - (s - bp)) + (lo - bp);
  const unsigned a = __float_as_uint(s);
  if ((a & 0xffffu) != 0x8000u || e == 0.0f) return bf_round(s);
  const float down = __uint_as_float(a & 0xffff0000u);            // toward zero
  const float up = __uint_as_float((a & 0xffff0000u) + 0x10000u);  // away from zero
  return ((e > 0.0f) == (s > 0.0f)) ? up : down;
}



// Wait for phase `parity` of an mbarrier, giving up after WAIT_LIMIT_CYCLES SM
// clock cycles (about a second; the SM cycle counter is far cheaper to read
// than %globaltimer).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long c0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity)) {
    if (clock64() - c0 > WAIT_LIMIT_CYCLES) return false;
  }
  return true;
}

// Mixed-precision fused multiply-adds (sm_100+): bf16 operands, fp32 sum.
// The bf16 x bf16 product is exact in fp32, so each call rounds once, as
// fmaf on the widened operands would, without converting them first.
__device__ __forceinline__ void fma_bf16_pair(unsigned a, unsigned b, float& lo, float& hi) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %1, ah, bh, %1;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "r"(a), "r"(b));
}
// As above for one product, the operands picked from halves AH / BH of packed words.
template <int AH, int BH>
__device__ __forceinline__ float fma_bf16(unsigned a, unsigned b, float c) {
  if constexpr (AH == 0 && BH == 0)
    asm("{\n\t.reg .b16 x0, x1, y0, y1;\n\tmov.b32 {x0, x1}, %1;\n\tmov.b32 {y0, y1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, x0, y0, %0;\n\t}" : "+f"(c) : "r"(a), "r"(b));
  else if constexpr (AH == 0 && BH == 1)
    asm("{\n\t.reg .b16 x0, x1, y0, y1;\n\tmov.b32 {x0, x1}, %1;\n\tmov.b32 {y0, y1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, x0, y1, %0;\n\t}" : "+f"(c) : "r"(a), "r"(b));
  else if constexpr (AH == 1 && BH == 0)
    asm("{\n\t.reg .b16 x0, x1, y0, y1;\n\tmov.b32 {x0, x1}, %1;\n\tmov.b32 {y0, y1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, x1, y0, %0;\n\t}" : "+f"(c) : "r"(a), "r"(b));
  else
    asm("{\n\t.reg .b16 x0, x1, y0, y1;\n\tmov.b32 {x0, x1}, %1;\n\tmov.b32 {y0, y1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, x1, y1, %0;\n\t}" : "+f"(c) : "r"(a), "r"(b));
  return c;
}
__device__ __forceinline__ float bf_bits(unsigned short x) { return __uint_as_float((unsigned)x << 16); }
__device__ __forceinline__ float bf_lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }

// ---- z = f_b . f_a ------------------------------------------------------------
// Lane l of warp w: group g = l >> 3 owns channels 16 w + 4 g + r (r = 0..3),
// kl = l & 7 owns k = 64 m + 8 kl + (0..7) (m = 0, 1); fbw[r][m] holds those
// 8 bf16 of the f_b row of channel r.  The lane sums the 16 exact products of
// each channel in two fp32 chains (even / odd k) and adds them; a reduce-
// scatter over the group's 8 lanes (offsets 4 and 2) and a full add at offset
// 1 leave channel row (l >> 1) & 3 on lanes l and l ^ 1.  No product passes
// more than 8 roundings in the lane and 3 in the tree, so
//   |z - exact| <= gamma_11 sum|p_j| <= 11 u (1 + 2^-10) |f_b row|_2 |f_a|_2
// (Cauchy-Schwarz, u = 2^-24); the bound used is 12 u (1 + 2^-10) times upper
// bounds of the two norms.
__device__ __forceinline__ void z_partials(const uint4 (&fbw)[4][2], const uint4 f0, const uint4 f1, float (&acc)[4]) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float lo = 0.0f, hi = 0.0f;
    fma_bf16_pair(fbw[r][0].x, f0.x, lo, hi);
    fma_bf16_pair(fbw[r][0].y, f0.y, lo, hi);
    fma_bf16_pair(fbw[r][0].z, f0.z, lo, hi);
    fma_bf16_pair(fbw[r][0].w, f0.w, lo, hi);
    fma_bf16_pair(fbw[r][1].x, f1.x, lo, hi);
    fma_bf16_pair(fbw[r][1].y, f1.y, lo, hi);
    fma_bf16_pair(fbw[r][1].z, f1.z, lo, hi);
    fma_bf16_pair(fbw[r][1].w, f1.w, lo, hi);
    acc[r] = lo + hi;
  }
}

__device__ __forceinline__ float z_reduce(const float (&acc)[4], int lane) {
  const bool b2 = (lane & 4) != 0, b1 = (lane & 2) != 0;
  float k0 = b2 ? acc[2] : acc[0], k1 = b2 ? acc[3] : acc[1];
  const float s0 = b2 ? acc[0] : acc[2], s1 = b2 ? acc[1] : acc[3];
  k0 += __shfl_xor_sync(0xffffffffu, s0, 4);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 4);
  float r = b1 ? k1 : k0;
  const float s = b1 ? k0 : k1;
  r += __shfl_xor_sync(0xffffffffu, s, 2);
  return r + __shfl_xor_sync(0xffffffffu, r, 1);
}

// z of one channel row of each lane group (the lane's 16 bf16 of it in w0, w1,
// of f_a in f0, f1), from its exact products summed as TwoSum pairs (Knuth)
// in the lane and across the group's 8 lanes; the pair hi + lo then rounds to
// the correctly rounded bf16 of z.  Every lane of the warp calls it together.
__device__ __forceinline__ float z_exact(const uint4 w0, const uint4 w1, const uint4 f0, const uint4 f1) {
  const unsigned w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  const unsigned fv[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
  float hi = 0.0f, lo = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float p = (j & 1) ? bf_hi(w[j >> 1]) * bf_hi(fv[j >> 1]) : bf_lo(w[j >> 1]) * bf_lo(fv[j >> 1]);
    const float s = hi + p, bp = s - hi;
    lo += (hi - (s - bp)) + (p - bp);
    hi = s;
  }
#pragma unroll
  for (int m = 1; m <= 4; m <<= 1) {
    const float ho = __shfl_xor_sync(0xffffffffu, hi, m);
    const float lo_o = __shfl_xor_sync(0xffffffffu, lo, m);
    const float s = hi + ho, bp = s - hi;
    lo = (lo + lo_o) + ((hi - (s - bp)) + (ho - bp));
    hi = s;
  }
  return bf16_round_pair(hi, lo);
}

// Row rs of fbw, picked by selects so that fbw is never indexed at run time
// (that would move it to local memory).
__device__ __forceinline__ unsigned pick4(int rs, unsigned a, unsigned b, unsigned c, unsigned d) {
  return rs < 2 ? (rs == 0 ? a : b) : (rs == 2 ? c : d);
}
__device__ __forceinline__ void fb_row(const uint4 (&fbw)[4][2], int rs, uint4& w0, uint4& w1) {
  w0.x = pick4(rs, fbw[0][0].x, fbw[1][0].x, fbw[2][0].x, fbw[3][0].x);
  w0.y = pick4(rs, fbw[0][0].y, fbw[1][0].y, fbw[2][0].y, fbw[3][0].y);
  w0.z = pick4(rs, fbw[0][0].z, fbw[1][0].z, fbw[2][0].z, fbw[3][0].z);
  w0.w = pick4(rs, fbw[0][0].w, fbw[1][0].w, fbw[2][0].w, fbw[3][0].w);
  w1.x = pick4(rs, fbw[0][1].x, fbw[1][1].x, fbw[2][1].x, fbw[3][1].x);
  w1.y = pick4(rs, fbw[0][1].y, fbw[1][1].y, fbw[2][1].y, fbw[3][1].y);
  w1.z = pick4(rs, fbw[0][1].z, fbw[1][1].z, fbw[2][1].z, fbw[3][1].z);
  w1.w = pick4(rs, fbw[0][1].w, fbw[1][1].w, fbw[2][1].w, fbw[3][1].w);
}

// ---- causal conv ----------------------------------------------------------------
// bf16 of SiLU(y), y = b + sum_k w_k s_k (four bf16 pairs), for the rare case in
// which the fast fp32 value lies too close to a rounding boundary.  First in
// fp32: y exactly as the pair s + e (TwoSum over the exact products), the
// sigmoid from expf (within 2 ulp) and an IEEE division; that settles most
// cases.  The rest go to fp64 (exact products and sums; the SiLU's own fp64
// error is far below a bf16 half ulp), which is slow on this part.
__device__ __forceinline__ float silu_bf16_exact(float b, unsigned wp0, unsigned wp1, unsigned s01, unsigned s23) {
  const float p[4] = {bf_lo(wp0) * bf_lo(s01), bf_hi(wp0) * bf_hi(s01), bf_lo(wp1) * bf_lo(s23),
                      bf_hi(wp1) * bf_hi(s23)};  // exact
  float sum = b, err = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float t = sum + p[k], bp = t - sum;
    err += (sum - (t - bp)) + (p[k] - bp);
    sum = t;
  }
  const float y = sum + err;  // within u |y| (1 + 4u) of the exact sum
  const float d = 1.0f + expf(-y);
  float sg = __frcp_rn(d);
  const float sy = fmaf(sum, sg, err * sg);
  // sigmoid: 2^-22 (expf) + u (1 + e^-y) + u (the reciprocal) + |y| u (the
  // error of y, through sigma' / sigma = 1 - sigma); the product one more u:
  // |sy - silu(exact y)| <= (2^-22 + 3u + |y| u) |sy|; margin x2
  if (fabsf(y) < 80.0f && !bf16_rounding_uncertain(sy, 2.0f * (0x1p-22f + (3.0f + fabsf(y)) * U32) * fabsf(sy)))
    return bf_round(sy);
  double yd = (double)b;
  yd = fma((double)bf_lo(wp0), (double)bf_lo(s01), yd);
  yd = fma((double)bf_hi(wp0), (double)bf_hi(s01), yd);
  yd = fma((double)bf_lo(wp1), (double)bf_lo(s23), yd);
  yd = fma((double)bf_hi(wp1), (double)bf_hi(s23), yd);
  return bf16_round_f64(yd * __drcp_rn(1.0 + exp(-yd)));  // y / (1 + e^-y) within 2 fp64 ulp
}
// The same out of line: with many tokens the unrolled conv is long enough for
// instruction fetch to matter, and the rare path is better kept out of it (up
// to four tokens the call's register saves cost more than the fetch).
__device__ __noinline__ float silu_bf16_exact_ool(float b, unsigned wp0, unsigned wp1, unsigned s01, unsigned s23) {
  return silu_bf16_exact(b, wp0, wp1, s01, s23);
}

// One channel over up to N tokens [t0, t0 + n): position p of the channel's
// input sequence is window slot p - (3 - SL) for p < 3 (the window right-
// aligned) and x_{p-3} from p = 3 on; taps are right-aligned in w[0..4) (zero
// taps in front when W < 4), so that y_t = b + sum_k w[k] seq(t + k).  The
// lane holds positions t0 .. t0 + N + 2 as raw bf16 bits, two to a word.
template <int N>
struct ConvLane {
  static constexpr int WORDS = (N + 4) / 2;
  unsigned sp[WORDS];  // position t0 + i in half i & 1 of word i >> 1
  unsigned wp[2];      // taps, w[k] in half k & 1 of word k >> 1
  unsigned short bb;   // bias
  __device__ __forceinline__ unsigned short get(int i) const {
    return (unsigned short)((i & 1) ? (sp[i >> 1] >> 16) : (sp[i >> 1] & 0xffffu));
  }
  __device__ __forceinline__ unsigned short tap(int k) const {
    return (unsigned short)((k & 1) ? (wp[k >> 1] >> 16) : (wp[k >> 1] & 0xffffu));
  }
};

// y = b + sum_k w[k] seq(i + k) for the lane's token i, each step rounded
// once; run collects |partial sums| (the fp32 error bound / u).
template <int I, int N>
__device__ __forceinline__ float conv_dot(const ConvLane<N>& q, float& run) {
  float y = bf_bits(q.bb);
  y = fma_bf16<0, (I & 1)>(q.wp[0], q.sp[I >> 1], y);
  run = fabsf(y);
  y = fma_bf16<1, ((I + 1) & 1)>(q.wp[0], q.sp[(I + 1) >> 1], y);
  run += fabsf(y);
  y = fma_bf16<0, ((I + 2) & 1)>(q.wp[1], q.sp[(I + 2) >> 1], y);
  run += fabsf(y);
  y = fma_bf16<1, ((I + 3) & 1)>(q.wp[1], q.sp[(I + 3) >> 1], y);
  run += fabsf(y);
  return y;
}

// Thread-block cluster helpers for the two-CTA split of a (request, head).
__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: writes before it are seen by reads after it.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 8 bytes of CTA `rank`'s shared memory at the address that `p` has in this CTA.
__device__ __forceinline__ uint2 ld_peer_u2(const void* p, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  uint2 v;
  asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(remote) : "memory");
  return v;
}
__device__ __forceinline__ int ld_peer_s32(const void* p, unsigned rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// DF: conv_state laid out [pool, 3D, W-1] (true) or [pool, W-1, 3D] (false).
// VS: the CTAs of a (request, head) -- 1, or 2 in a cluster, each owning 64 of the 128
// v rows (one pass of the recurrence) and half of the outputs; both run the prologue
// and swap their halves of o through distributed shared memory for the RMSNorm.
template <int L, bool BS, bool DF, int VS>
__global__ void __launch_bounds__(THREADS, (L <= 4 ? 3 : 2)) kda_step_kernel(const StepArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using S = Smem<L, BS>;
  using SB = StateT<BS>;
  unsigned char* stc = smem + S::state;  // the state in its storage type
  float* st = reinterpret_cast<float*>(stc);
  unsigned short* stb = reinterpret_cast<unsigned short*>(stc);
  float* eg = reinterpret_cast<float*>(smem + S::eg);
  float* kh = reinterpret_cast<float*>(smem + S::kh);
  float* qh = reinterpret_cast<float*>(smem + S::qh);
  unsigned short* fa_b = reinterpret_cast<unsigned short*>(smem + S::fa);
  __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(smem + S::fa);  // reuses the f_a space
  __nv_bfloat16* vv = reinterpret_cast<__nv_bfloat16*>(smem + S::vv);
  __half* gsig_s = reinterpret_cast<__half*>(smem + S::gate);  // sigmoid of the out-gate
  float* fnp = reinterpret_cast<float*>(smem + S::fnp);
  float* beta_s = reinterpret_cast<float*>(smem + S::beta);
  float* kq_s = reinterpret_cast<float*>(smem + S::kq);
  int* slot_s = reinterpret_cast<int*>(smem + S::slot);
  int* ctl = reinterpret_cast<int*>(smem + S::ctl);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S::mbar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  static_assert(VS == 1 || VS == 2, "one or two CTAs a (request, head)");
  const unsigned slice = VS == 1 ? 0u : cluster_rank();  // which 64 v rows (VS = 2)
  const unsigned task = blockIdx.x / VS;                // the clusters of a launch are consecutive blocks
  const int h = (int)(task % (unsigned)a.heads);        // 32-bit: a 64-bit division costs every CTA
  const long long r = task / (unsigned)a.heads;
  const long long row0 = r * L;
  const int D = a.D, SL = a.W - 1;

  // ---- round trip 1: everything that needs no other value -------------------
  int sl[L];
#pragma unroll
  for (int t = 0; t < L; ++t) sl[t] = a.slots[row0 + t];
  const int acc = (a.accepted != nullptr) ? a.accepted[r] : 1;
  // z operands of the lane's 4 channels (see z_partials)
  const int zc = warp * Z_CHANNELS + (lane >> 3) * 4 + ((lane >> 1) & 3);  // channel of the lane's z
  uint4 fbw[4][2];
  {
    const uint4* fb = reinterpret_cast<const uint4*>(a.f_b + (long long)(h * HD + warp * Z_CHANNELS + (lane >> 3) * 4) * HD);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
      for (int m = 0; m < 2; ++m) fbw[rr][m] = __ldg(fb + rr * (HD / 8) + m * 8 + (lane & 7));
  }
  const float fbn = a.fb_norm[h * HD + zc];  // |f_b row|_2, rounded up
  const float dtc = a.dt_bias[h * HD + zc];
  const float a_log = a.A_log[h];
  // Launched as a programmatic dependent of the projection that writes
  // `projected` (a layer plan), the loads above -- weights, slots -- overlap
  // that kernel's tail; from here on its output is read. Without such a
  // dependency this returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // f_a and out-gate of the L tokens, raw bf16
  constexpr int PER_THREAD = (L * HD + THREADS - 1) / THREADS;
  unsigned short fa_v[PER_THREAD], gate_v[PER_THREAD];
#pragma unroll
  for (int i = 0; i < PER_THREAD; ++i) {
    const int e = tid + i * THREADS;
    fa_v[i] = gate_v[i] = 0;
    if (e < L * HD) {
      const unsigned short* prow = reinterpret_cast<const unsigned short*>(a.projected + (row0 + e / HD) * a.pitch);
      fa_v[i] = prow[4 * D + (e % HD)];
      gate_v[i] = prow[3 * D + h * HD + (e % HD)];
    }
  }
  float beta_logit = 0.0f;
  if (tid < L) beta_logit = bf(a.projected[(row0 + tid) * a.pitch + 4 * D + HD + h]);

  // conv work: channel c of the head; the first half of the CTA takes q and k
  // over tokens [0, A) and v over [0, B), the second half q and k over [A, L)
  // and v over [B, L) (A = ceil(L/2), B = floor(L/2)): 1.5 L outputs a thread
  // for even L.  One code path serves both halves (a second copy of the conv
  // costs more in instruction fetch than its constant token offsets save).
  constexpr int CA = (L + 1) / 2, CB = L / 2;
  const int c = tid & (HD - 1);
  const bool second = tid >= HD;
  // first token and token count of kind 0, 1 (q, k) and 2 (v)
  auto conv_t0 = [&](int kind) { return (kind < 2) ? (second ? CA : 0) : (second ? CB : 0); };
  auto conv_n = [&](int kind) { return (kind < 2) ? (second ? L - CA : CA) : (second ? L - CB : CB); };
  ConvLane<CA> cv[3];
#pragma unroll
  for (int kind = 0; kind < 3; ++kind) {
    const uint2 wt = a.conv_w[kind * D + h * HD + c];
    cv[kind].wp[0] = wt.x;
    cv[kind].wp[1] = wt.y;
    cv[kind].bb = a.bias ? reinterpret_cast<const unsigned short*>(a.bias)[kind * D + h * HD + c] : (unsigned short)0;
  }
  // The conv inputs from the projected rows (sequence positions 3 on) need no slot.
  // Decode's (one a channel) go out with round trip 1, the start window below them
  // waiting for the slots (large decode 127.3 -> 124.9 us); verify's, several a
  // channel, go out with the window in round trip 2 (issued here they delayed round
  // trip 1: spec-verify 24.7 -> 25.3 us).
  constexpr bool EARLY_X = (L == 1);
  unsigned short xin[3][CA + 3];
  if constexpr (EARLY_X) {
    const unsigned short* prow =
        reinterpret_cast<const unsigned short*>(a.projected) + row0 * a.pitch + h * HD + c;
#pragma unroll
    for (int kind = 0; kind < 3; ++kind) {
      const int t0 = conv_t0(kind), n = conv_n(kind);
#pragma unroll
      for (int i = 0; i < CA + 3; ++i) {
        const int pos = t0 + i;  // sequence position; pos - 3 < t0 + n <= L
        xin[kind][i] = (n > 0 && i < n + 3 && pos >= 3) ? prow[(long long)(pos - 3) * a.pitch + kind * D]
                                                        : (unsigned short)0;
      }
    }
  }

  // ---- validate (every thread decides the same from the same loaded values) ---
  int status = TASK_OK, start = 0;
  if (sl[0] == -1) {
    status = TASK_PADDING;
  } else if (acc < 1 || acc > L) {
    status = TASK_SKIP;
    if (tid == 0) atomicOr(a.err, KDA_ERR_ACCEPTED);
  } else {
    bool bad = false;
#pragma unroll
    for (int t = 0; t < L; ++t) {
      bad |= (sl[t] < 0) || (sl[t] >= a.pool);
      start |= sl[t] & (0 - (int)(t == acc - 1));  // sl[acc - 1] without a run-time index
    }
    if (bad) {
      status = TASK_SKIP;
      if (tid == 0) atomicOr(a.err, KDA_ERR_SLOT);
    }
  }
  if (status == TASK_PADDING) {  // zero output rows (this CTA's columns), no cache traffic
    constexpr int CW = HD / VS;
    for (int i = tid; i < L * CW; i += THREADS)
      a.out[(row0 + i / CW) * D + h * HD + slice * CW + (i % CW)] = __float2bfloat16_rn(0.0f);
    return;
  }
  if (status != TASK_OK) return;

  // ---- round trip 2: the conv inputs, then the start state (bulk) -------------
  // The start window of the thread's channels (sequence positions below 3; verify:
  // and the projected x above it) goes out first so that it does not queue behind
  // the state's bulk copies; the conv inputs are packed once the copies are issued.
  // Conv cache addressing (elements): slot s, channel ch, window slot j at
  // s * slot_elems + ch * CHS + j * JS.
  const long long slot_elems = 3LL * D * SL;
  const long long CHS = DF ? SL : 1, JS = DF ? 1 : 3LL * D;
  // the thread's q channel: column h * 128 + c; k and v are D and 2 D further
  const long long cch = (long long)(h * HD + c) * CHS;
  if constexpr (EARLY_X) {  // the start window alone
    const unsigned short* win =
        reinterpret_cast<const unsigned short*>(a.conv_state) + (long long)start * slot_elems + cch;
#pragma unroll
    for (int kind = 0; kind < 3; ++kind) {
      const int t0 = conv_t0(kind), n = conv_n(kind);
#pragma unroll
      for (int i = 0; i < 3; ++i) {  // positions t0 + i < 3 only
        const int pos = t0 + i;
        const int j = pos + SL - 3;  // window slot of the position
        if (n > 0 && pos < 3 && j >= 0) xin[kind][i] = win[(long long)kind * D * CHS + j * JS];
      }
    }
  } else {  // projected x and the start window together
    const unsigned short* prow =
        reinterpret_cast<const unsigned short*>(a.projected) + row0 * a.pitch + h * HD + c;
    const unsigned short* win =
        reinterpret_cast<const unsigned short*>(a.conv_state) + (long long)start * slot_elems + cch;
#pragma unroll
    for (int kind = 0; kind < 3; ++kind) {
      const int t0 = conv_t0(kind), n = conv_n(kind);
#pragma unroll
      for (int i = 0; i < CA + 3; ++i) {
        const int pos = t0 + i;  // sequence position; pos - 3 < t0 + n <= L
        unsigned short v = 0;
        if (n > 0 && i < n + 3) {
          if (pos >= 3) {
            v = prow[(long long)(pos - 3) * a.pitch + kind * D];
          } else {
            const int j = pos + SL - 3;  // window slot of the position
            if (j >= 0) v = win[(long long)kind * D * CHS + j * JS];
          }
        }
        xin[kind][i] = v;
      }
    }
  }
  // Decode (many CTAs a SM, one after another) puts the state in flight at
  // once; verify (often a single wave of CTAs, all in this phase together)
  // first waits for the conv inputs, which would otherwise queue behind every
  // CTA's state copies, and has its conv and gates to cover the state's latency.
  const int Q0 = (int)slice * (QUARTERS / VS);  // this CTA's first quarter of the state
  auto issue_state = [&]() {
    if (tid == 0) {
      const unsigned char* src = static_cast<const unsigned char*>(a.state_pool) +
                                 ((long long)start * a.heads + h) * SB::BYTES;
#pragma unroll
      for (int q = 0; q < QUARTERS; ++q) mbar_init(smem_u32(&mbar[q]), 1);
      fence_mbar_init();
#pragma unroll
      for (int q = Q0; q < Q0 + QUARTERS / VS; ++q) {  // this CTA's quarters
        const uint32_t bar = smem_u32(&mbar[q]);
        mbar_expect_tx(bar, SB::QBYTES);
        bulk_load(smem_u32(stc + q * SB::QBYTES), src + q * SB::QBYTES, SB::QBYTES, bar);
      }
      ctl[0] = 0;
    }
  };
  if constexpr (L == 1) issue_state();
#pragma unroll
  for (int t = 0; t < L; ++t)
    if (tid == t) slot_s[t] = sl[t];
#pragma unroll
  for (int i = 0; i < PER_THREAD; ++i) {
    const int e = tid + i * THREADS;
    if ((tid & ~31) + i * THREADS < L * HD) {  // warp-uniform
      fa_b[e] = fa_v[i];
      gsig_s[e] = __float2half_rn(sigmoid_fast(bf_bits(gate_v[i])));  // within 2^-11 relative; the output is bf16
      // squares of f_a: one partial sum per (token, 32 channels)
      const float f = bf_bits(fa_v[i]);
      const float sq = warp_sum(f * f);
      if (lane == 0) fnp[(e / HD) * 4 + (e % HD) / 32] = sq;
    }
  }
  if (tid < L) beta_s[tid] = sigmoid_fast(beta_logit);
#pragma unroll
  for (int kind = 0; kind < 3; ++kind)
#pragma unroll
    for (int w = 0; w < ConvLane<CA>::WORDS; ++w)
      cv[kind].sp[w] = xin[kind][2 * w] | ((2 * w + 1 < CA + 3) ? ((unsigned)xin[kind][2 * w + 1] << 16) : 0u);
  if constexpr (L > 1) {
    // thread 0 issues the copies only once its own conv inputs are in
    asm volatile("" ::"r"(cv[0].sp[0] | cv[1].sp[0] | cv[2].sp[0]));
    issue_state();
  }
  __syncthreads();  // barriers initialised, f_a, its squares and the slots staged

  // ---- causal conv of the thread's channels (correctly rounded) ---------------
  // It runs before z: its inputs arrived with round trips 1 and 2, which the
  // recurrence waits for anyway, and they are dead before z needs registers.
  {
#pragma unroll
    for (int kind = 0; kind < 3; ++kind) {
      const ConvLane<CA>& q = cv[kind];
      const int t0 = conv_t0(kind), n = conv_n(kind);
#pragma unroll
      for (int i = 0; i < CA; ++i) {
        if (i >= n) continue;
        const int t = t0 + i;
        float run;  // sum of |partial sums|, the fp32 error bound / u
        float y;
        switch (i) {  // compile-time after unrolling
          case 0: y = conv_dot<0>(q, run); break;
          case 1: y = conv_dot<1>(q, run); break;
          case 2: y = conv_dot<2>(q, run); break;
          default: y = conv_dot<3>(q, run); break;
        }
        const float sy = y * sigmoid_fast(y);  // SiLU
        // |y - exact| <= 1.1 u run and SiLU' <= 1.1; the sigmoid and the
        // product add at most (2.35 |y| u + 2^-21 + 2u) |sy|:
        // |sy - silu(exact y)| <= 1.21 u run + (2.5 u |y| + 2^-20) |sy|; margin x2
        float yb;
        if (!bf16_rounding_uncertain(sy, 2.0f * (1.21f * U32 * run + (2.5f * U32 * fabsf(y) + 0x1p-20f) * fabsf(sy)))) {
          yb = bf_round(sy);
        } else {
          const unsigned s01 = q.get(i) | ((unsigned)q.get(i + 1) << 16);
          const unsigned s23 = q.get(i + 2) | ((unsigned)q.get(i + 3) << 16);
          if constexpr (L > 4) yb = silu_bf16_exact_ool(bf_bits(q.bb), q.wp[0], q.wp[1], s01, s23);
          else yb = silu_bf16_exact(bf_bits(q.bb), q.wp[0], q.wp[1], s01, s23);
        }
        if (kind == 0) qh[t * HD + c] = yb;
        else if (kind == 1) kh[t * HD + c] = yb;
        else vv[t * HD + c] = __float2bfloat16_rn(yb);
      }
    }
  }
  // The windows after each token (copies of the conv inputs, still in the
  // thread's registers) go out after z and the l2norm: scattered 2-byte stores
  // queue in the SM's memory pipeline, and shuffles and shared-memory loads
  // issued behind them wait until they drain.
  auto store_windows = [&]() {
    unsigned short* conv16 = reinterpret_cast<unsigned short*>(a.conv_state);
#pragma unroll
    for (int kind = 0; kind < 3; ++kind) {
      const ConvLane<CA>& q = cv[kind];
      const int t0 = conv_t0(kind), n = conv_n(kind);
      // sequence position t + p (p = 1..3) goes to window slot p + SL - 4 of slots[r, t]
      const long long wk = cch + (long long)kind * D * CHS + (long long)(SL - 4) * JS;
#pragma unroll
      for (int i = 0; i < CA; ++i) {
        if (i >= n) continue;
        const long long cb = wk + (long long)slot_s[t0 + i] * slot_elems;
#pragma unroll
        for (int p = 1; p <= 3; ++p)
          if (p + SL >= 4) conv16[cb + p * JS] = q.get(i + p);
      }
    }
  };
  // ---- z = f_b . f_a (correctly rounded), lower-bound gate, e^g ---------------
  {
    const float expA = expf(a_log);
    // unrolled for short verifies; rolled above four tokens (instruction fetch)
#pragma unroll(L <= 4 ? 2 : 1)
    for (int t = 0; t < L; t += 2) {
      const bool pair = (t + 1 < L);
      const uint4* f0 = reinterpret_cast<const uint4*>(fa_b + t * HD);
      float p0[4];
      z_partials(fbw, f0[lane & 7], f0[8 + (lane & 7)], p0);
      float z = z_reduce(p0, lane);
      int tt = t;
      if (pair) {
        const uint4* f1 = reinterpret_cast<const uint4*>(fa_b + (t + 1) * HD);
        float p1[4];
        z_partials(fbw, f1[lane & 7], f1[8 + (lane & 7)], p1);
        const float z1 = z_reduce(p1, lane);
        if (lane & 1) {  // odd lanes finish token t + 1, even lanes token t
          z = z1;
          tt = t + 1;
        }
      }
      // |f_a|_2 of token tt, rounded up: the fp32 sum of 128 squares is within
      // 2^-17 relative of exact, its root within 2^-18 + 2^-21
      const float4 np = *reinterpret_cast<const float4*>(fnp + tt * 4);
      const float fnorm = sqrt_fast((np.x + np.y) + (np.z + np.w)) * (1.0f + 0x1p-12f);
      const float bound = 12.0f * U32 * (1.0f + 0x1p-10f) * fbn * fnorm;
      const bool unsure = bf16_rounding_uncertain(z, bound);
      unsigned redo = __ballot_sync(0xffffffffu, unsure) & (pair ? 0xffffffffu : 0x55555555u);
      z = bf_round(z);
      // Each 8-lane group resolves its own first undecided lane per round (the
      // exact sum runs within a group), so a round settles up to four.
      const int g8 = lane & 24;
      while (redo) {
        const unsigned mine = (redo >> g8) & 0xffu;
        const int li = g8 + (mine ? __ffs(mine) - 1 : 0);
        redo &= ~__ballot_sync(0xffffffffu, mine != 0 && lane == li);
        const uint4* fr = reinterpret_cast<const uint4*>(fa_b + (pair ? t + (li & 1) : t) * HD);
        uint4 w0, w1;
        fb_row(fbw, (li >> 1) & 3, w0, w1);
        const float ex = z_exact(w0, w1, fr[lane & 7], fr[8 + (lane & 7)]);
        if (mine != 0 && lane == li) z = ex;
      }
      if (pair || (lane & 1) == 0) {
        const float x = z + dtc;
        const float g = (a.gate_mode == KDA_GATE_SOFTPLUS) ? fmaxf(-expA * softplus_fast(x), a.lb)
                                                          : a.lb * sigmoid_fast(expA * x);
        eg[tt * HD + zc] = __expf(g);
      }
    }
  }

  __syncthreads();  // raw q, k, v and e^g of every channel written

  // ---- l2norm of q and k, k^.q^: warp t on token t ----------------------------------
  // Each warp reads and rewrites its own token only; the other warps go on to
  // the barrier.
  if (warp < L) {
    const int t = warp;
    float4 q = *reinterpret_cast<float4*>(qh + t * HD + lane * 4);
    float4 k = *reinterpret_cast<float4*>(kh + t * HD + lane * 4);
    const float sq = warp_sum(q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
    const float sk = warp_sum(k.x * k.x + k.y * k.y + k.z * k.z + k.w * k.w);
    const float sqk = warp_sum(q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w);
    const float rq = rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
    const float fq = rq * a.q_scale;
    q.x *= fq; q.y *= fq; q.z *= fq; q.w *= fq;
    k.x *= rk; k.y *= rk; k.z *= rk; k.w *= rk;
    *reinterpret_cast<float4*>(qh + t * HD + lane * 4) = q;
    *reinterpret_cast<float4*>(kh + t * HD + lane * 4) = k;
    if (lane == 0) kq_s[t] = sqk * fq * rk;
  }
  __syncthreads();
  if constexpr (VS == 2) {
    // Both CTAs read the start window, and it may be one of the windows written
    // below: the other CTA's conv inputs are in its registers before slice 0 stores.
    cluster_barrier();
  }
  if (VS == 1 || slice == 0) store_windows();  // the windows once per (request, head)

  // ---- recurrence: 2 passes of 2 quarters; 16 lanes per v row, 8 k values a lane --
  // Lane l: half hs = l >> 4 of the warp, kl = l & 15 owns k = 64 m + 4 kl + (0..3)
  // (m = 0, 1); in pass p the thread holds rows 64 p + 32 (r >> 1) + 16 (r & 1) +
  // 2 warp + hs (r = 0..3), i.e. one row of each quarter half.  A warp half
  // reads each k-slice of e^g, q^, k^ once per token.
  const int hs = lane >> 4, kl = lane & 15;
  const int rbase = warp * 2 + hs;
  const bool b3 = (kl & 8) != 0, b2 = (kl & 4) != 0, b1 = (kl & 2) != 0;
  const int rsel = (b2 ? 2 : 0) + (b1 ? 1 : 0);  // row of the value this lane ends with
  bool timed_out = false;
  // element (h, row, 64 m + 4 kl) of a slot's state, in bytes from the slot's block
  unsigned char* dst_k = static_cast<unsigned char*>(a.state_pool) + ((long long)h * STATE_FLOATS + kl * 4) * SB::ELEM;
#pragma unroll 1
  for (int pass = (int)slice; pass < (int)slice + 2 / VS; ++pass) {  // VS = 2: the CTA's one pass
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&mbar[2 * pass]), 0) &&
                                                mbar_wait_bounded(smem_u32(&mbar[2 * pass + 1]), 0));
    if (!ok) timed_out = true;
    if (ok) {
    // 4 rows, 8 k values each as 4 float2 pairs
    float2 sv[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int row = pass * 64 + (r >> 1) * 32 + (r & 1) * 16 + rbase;
        if constexpr (BS) {  // four bf16, widened exactly
          const uint2 x = *reinterpret_cast<const uint2*>(stb + row * HD + m * 64 + kl * 4);
          sv[r][2 * m] = make_float2(bf_lo(x.x), bf_hi(x.x));
          sv[r][2 * m + 1] = make_float2(bf_lo(x.y), bf_hi(x.y));
        } else {
          const float4 x = *reinterpret_cast<const float4*>(st + row * HD + m * 64 + kl * 4);
          sv[r][2 * m] = make_float2(x.x, x.y);
          sv[r][2 * m + 1] = make_float2(x.z, x.w);
        }
      }
    const int vq = pass * 64 + (rsel >> 1) * 32 + (rsel & 1) * 16 + rbase;  // row of this lane's value
#pragma unroll 1
    for (int t = 0; t < L; ++t) {
      float2 kv[4], dk2[4], dq2[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) dk2[r] = dq2[r] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int k0 = t * HD + m * 64 + kl * 4;
        const float4 e = *reinterpret_cast<const float4*>(eg + k0);
        const float4 qv = *reinterpret_cast<const float4*>(qh + k0);
        const float4 k4 = *reinterpret_cast<const float4*>(kh + k0);
        const float2 e0 = make_float2(e.x, e.y), e1 = make_float2(e.z, e.w);
        const float2 q0 = make_float2(qv.x, qv.y), q1 = make_float2(qv.z, qv.w);
        kv[2 * m] = make_float2(k4.x, k4.y);
        kv[2 * m + 1] = make_float2(k4.z, k4.w);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          sv[r][2 * m] = mul2(sv[r][2 * m], e0);  // S' = diag(e^g) S
          sv[r][2 * m + 1] = mul2(sv[r][2 * m + 1], e1);
          dk2[r] = fma2(sv[r][2 * m], kv[2 * m], dk2[r]);
          dk2[r] = fma2(sv[r][2 * m + 1], kv[2 * m + 1], dk2[r]);
          dq2[r] = fma2(sv[r][2 * m], q0, dq2[r]);
          dq2[r] = fma2(sv[r][2 * m + 1], q1, dq2[r]);
        }
      }
      // reduce-scatter of S'^T k^ and S'^T q^ of the 4 rows over the row's 16
      // lanes (offsets 8, 4, 2, then a full add at 1): lane kl ends with
      // S'^T k^ (kl < 8) or S'^T q^ (kl >= 8) of row rsel, on lanes kl and kl ^ 1
      float v8[8];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        v8[r] = dk2[r].x + dk2[r].y;
        v8[4 + r] = dq2[r].x + dq2[r].y;
      }
      float w4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float keep = b3 ? v8[4 + i] : v8[i], send = b3 ? v8[i] : v8[4 + i];
        w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
      }
      float w2[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float keep = b2 ? w4[2 + i] : w4[i], send = b2 ? w4[i] : w4[2 + i];
        w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
      float rv = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
      rv += __shfl_xor_sync(0xffffffffu, rv, 1);
      // beta u = beta (v - S'^T k^) on the lanes holding S'^T k^, then to the half
      const float bt = beta_s[t];
      const float bu_own = bt * (bf(vv[t * HD + vq]) - rv);
      const int src = lane & 16;
      float bu[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) bu[r] = __shfl_sync(0xffffffffu, bu_own, src | (2 * r));
      if (b3 && (kl & 1) == 0) {  // S_new^T q^ = S'^T q^ + beta u (k^.q^)
        const float bur = b2 ? (b1 ? bu[3] : bu[2]) : (b1 ? bu[1] : bu[0]);
        ob[t * HD + vq] = __float2bfloat16_rn(fmaf(bur, kq_s[t], rv));
      }
      unsigned char* dst = dst_k + (long long)slot_s[t] * a.heads * SB::BYTES;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = pass * 64 + (r >> 1) * 32 + (r & 1) * 16 + rbase;
        const float2 bu2 = make_float2(bu[r], bu[r]);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          sv[r][2 * m] = fma2(bu2, kv[2 * m], sv[r][2 * m]);  // S += beta k^ u^T
          sv[r][2 * m + 1] = fma2(bu2, kv[2 * m + 1], sv[r][2 * m + 1]);
          const float4 row4 = make_float4(sv[r][2 * m].x, sv[r][2 * m].y, sv[r][2 * m + 1].x, sv[r][2 * m + 1].y);
          if constexpr (BS) {  // rounded to bf16 (nearest even) as it is stored
            const uint2 w = make_uint2(pack_bf16x2(row4.x, row4.y), pack_bf16x2(row4.z, row4.w));
            store_streaming_u2(dst + (row * HD + m * 64) * 2, w);
          } else {
            store_streaming(reinterpret_cast<float*>(dst + (row * HD + m * 64) * 4), row4);
          }
        }
      }
    }
    }  // ok
  }
  // a dependent launch (the o_proj of a layer plan) may start its CTAs now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the RMSNorm weights of this lane, in flight across the barrier
  const float4 onw = *reinterpret_cast<const float4*>(a.o_norm + lane * 4);
  if (timed_out && lane == 0) {
    ctl[0] = 1;
    atomicOr(a.err, KDA_ERR_TIMEOUT);
  }
  __syncthreads();
  if constexpr (VS == 2) {
    // Both CTAs reach both cluster barriers, timed out or not. The first makes each
    // CTA's half of o (and its timeout flag) visible to the other; each then copies the
    // other's half into its own o; the second keeps each CTA's shared memory until the
    // other has read it.
    cluster_barrier();
    const unsigned peer = slice ^ 1u;
    constexpr int HALF = HD / 2;
    for (int i = tid; i < L * HALF / 4; i += THREADS) {  // 4 bf16 a load
      const int t = i / (HALF / 4), c = (int)peer * HALF + (i % (HALF / 4)) * 4;
      *reinterpret_cast<uint2*>(ob + t * HD + c) = ld_peer_u2(ob + t * HD + c, peer);
    }
    const int peer_timeout = (tid == 0) ? ld_peer_s32(ctl, peer) : 0;
    cluster_barrier();
    if (tid == 0 && peer_timeout) ctl[0] = 1;  // either half timed out: the request's outputs are not written
    __syncthreads();
  }
  if (ctl[0] != 0) {
    // Give copies still in flight a second bounded chance to land before the
    // shared memory is released; the outputs of this request stay unwritten.
    if (tid == 0) {
      for (int q = Q0; q < Q0 + QUARTERS / VS; ++q) (void)mbar_wait_bounded(smem_u32(&mbar[q]), 0);
    }
    return;
  }

  // ---- gated RMSNorm: warp t on token t; the other warps are done ------------------
  if (warp >= L) return;
  {
    const int t = warp;
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = bf(ob[t * HD + lane * 4 + e]);
    const float ss = warp_sum(o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3]);
    const float rstd = rsqrtf(ss * (1.0f / HD) + a.eps);
    const float wn[4] = {onw.x, onw.y, onw.z, onw.w};
    __align__(8) __nv_bfloat16 y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      y[e] = __float2bfloat16_rn(o[e] * rstd * wn[e] * __half2float(gsig_s[t * HD + lane * 4 + e]));
    if (VS == 1 || (unsigned)(lane >> 4) == slice)  // VS = 2: this CTA's 64 columns
      *reinterpret_cast<uint2*>(a.out + (row0 + t) * D + h * HD + lane * 4) = *reinterpret_cast<uint2*>(y);
  }
}

// ---- decode: two rows of one head a CTA -----------------------------------------------
// A one-row CTA spends much of its life on its two dependent load round trips
// (the slot, then the window and state it addresses). A CTA that serves rows 2p
// and 2p + 1 of head h shares those round trips and the head's f_b between the
// rows. With a bf16 pool the two 32 KiB states take the shared memory one fp32
// state takes; with an fp32 pool the second row's state halves are loaded into
// the one 64 KiB buffer as each of the first row's passes has taken its half
// into registers (a barrier a pass of the first row), so the second row's copies
// run under the first row's work. Three CTAs an SM either way. The arithmetic of
// a row is the one-row kernel's: thread half t runs row t's conv (q, k and v of
// its channel), z takes the two rows as a verify takes two tokens, warp t runs
// row t's norms, and each row's state goes through two passes of its own. The
// new state rows leave straight from registers as streaming stores, as in the
// one-row kernel: with four passes a CTA, the barrier a pass that a shared-memory
// write-back and bulk store need cost more than the stores save (bf16 pool, large
// decode: 79.6 us with bulk stores, 73.4 without).
template <bool BS>
struct SmemPair {
  // bf16: one [128][128] state a row; fp32: one [128][128] state, the second row's
  // halves loaded into it as the first row's passes free them
  static constexpr int state = 0;
  static constexpr int eg = state + (BS ? 2 * StateT<true>::BYTES : StateT<false>::BYTES);  // float [2][128]
  static constexpr int kh = eg + 2 * HD * 4;                   // float [2][128]   k, then k^
  static constexpr int qh = kh + 2 * HD * 4;                   // float [2][128]   q, then q^
  static constexpr int fa = qh + 2 * HD * 4;                   // bf16  [2][128]   f_a; later o
  static constexpr int vv = fa + 2 * HD * 2;                   // bf16  [2][128]
  static constexpr int gate = vv + 2 * HD * 2;                 // fp16  [2][128]   sigmoid(out-gate)
  static constexpr int fnp = gate + 2 * HD * 2;                // float [2][4]
  static constexpr int beta = fnp + 32;                        // float [2]
  static constexpr int kq = beta + 8;                          // float [2]
  static constexpr int slot = kq + 8;                          // int   [2]
  static constexpr int ctl = slot + 8;                         // int   [2]
  static constexpr int mbar = (ctl + 8 + 7) / 8 * 8;           // u64   [2][4]
  static constexpr int bytes = mbar + 8 * 2 * QUARTERS;
};

template <bool BS, bool DF>
__global__ void __launch_bounds__(THREADS, 3) kda_decode_pair_kernel(const StepArgs a, int rows) {
  extern __shared__ __align__(128) unsigned char smem[];
  using S = SmemPair<BS>;
  using SB = StateT<BS>;
  unsigned short* stb = reinterpret_cast<unsigned short*>(smem + S::state);
  float* st = reinterpret_cast<float*>(smem + S::state);
  float* eg = reinterpret_cast<float*>(smem + S::eg);
  float* kh = reinterpret_cast<float*>(smem + S::kh);
  float* qh = reinterpret_cast<float*>(smem + S::qh);
  unsigned short* fa_b = reinterpret_cast<unsigned short*>(smem + S::fa);
  __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(smem + S::fa);  // reuses the f_a space
  __nv_bfloat16* vv = reinterpret_cast<__nv_bfloat16*>(smem + S::vv);
  __half* gsig_s = reinterpret_cast<__half*>(smem + S::gate);
  float* fnp = reinterpret_cast<float*>(smem + S::fnp);
  float* beta_s = reinterpret_cast<float*>(smem + S::beta);
  float* kq_s = reinterpret_cast<float*>(smem + S::kq);
  int* slot_s = reinterpret_cast<int*>(smem + S::slot);
  int* ctl = reinterpret_cast<int*>(smem + S::ctl);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S::mbar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned task = blockIdx.x;
  const int h = (int)(task % (unsigned)a.heads);
  const long long row0 = 2LL * (task / (unsigned)a.heads);
  const int nrow = (row0 + 1 < rows) ? 2 : 1;
  const int D = a.D, SL = a.W - 1;
  const int c = tid & (HD - 1), my = tid >> 7;  // the thread's channel and row for the conv

  // ---- round trip 1 -----------------------------------------------------------------
  const int sl0 = a.slots[row0];
  const int sl1 = nrow == 2 ? a.slots[row0 + 1] : -1;
  const int zc = warp * Z_CHANNELS + (lane >> 3) * 4 + ((lane >> 1) & 3);
  uint4 fbw[4][2];
  {
    const uint4* fb = reinterpret_cast<const uint4*>(a.f_b + (long long)(h * HD + warp * Z_CHANNELS + (lane >> 3) * 4) * HD);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
      for (int m = 0; m < 2; ++m) fbw[rr][m] = __ldg(fb + rr * (HD / 8) + m * 8 + (lane & 7));
  }
  const float fbn = a.fb_norm[h * HD + zc];
  const float dtc = a.dt_bias[h * HD + zc];
  const float a_log = a.A_log[h];
  asm volatile("griddepcontrol.wait;" ::: "memory");  // as in the one-row kernel
  unsigned short fa_v = 0, gate_v = 0;
  const unsigned short* prow = reinterpret_cast<const unsigned short*>(a.projected) + (row0 + my) * a.pitch;
  if (my < nrow) {
    fa_v = prow[4 * D + c];
    gate_v = prow[3 * D + h * HD + c];
  }
  float beta_logit = 0.0f;
  if (tid < nrow) beta_logit = bf(a.projected[(row0 + tid) * a.pitch + 4 * D + HD + h]);
  ConvLane<1> cv[3];
  unsigned short xin[3][4];
#pragma unroll
  for (int kind = 0; kind < 3; ++kind) {
    const uint2 wt = a.conv_w[kind * D + h * HD + c];
    cv[kind].wp[0] = wt.x;
    cv[kind].wp[1] = wt.y;
    cv[kind].bb = a.bias ? reinterpret_cast<const unsigned short*>(a.bias)[kind * D + h * HD + c] : (unsigned short)0;
    xin[kind][0] = xin[kind][1] = xin[kind][2] = 0;
    xin[kind][3] = my < nrow ? prow[kind * D + h * HD + c] : (unsigned short)0;
  }

  // ---- validate each row (every thread decides the same) ------------------------------
  constexpr int TASK_NONE = 3;  // past the last row
  const int sl[2] = {sl0, sl1};
  int status[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    if (t >= nrow) status[t] = TASK_NONE;
    else if (sl[t] == -1) status[t] = TASK_PADDING;
    else if (sl[t] < 0 || sl[t] >= a.pool) status[t] = TASK_SKIP;
    else status[t] = TASK_OK;
  }
  // row t's status without a run-time index into the array
  auto row_ok = [&](int t) { return (t == 0 ? status[0] : status[1]) == TASK_OK; };
  if (tid == 0 && (status[0] == TASK_SKIP || status[1] == TASK_SKIP)) atomicOr(a.err, KDA_ERR_SLOT);
#pragma unroll
  for (int t = 0; t < 2; ++t)  // padding rows: zero output columns, no cache traffic
    if (status[t] == TASK_PADDING && my == t) a.out[(row0 + t) * D + h * HD + c] = __float2bfloat16_rn(0.0f);
  if (status[0] != TASK_OK && status[1] != TASK_OK) return;

  // ---- round trip 2: the start window of the thread's row, then the states (bulk) -----
  const long long slot_elems = 3LL * D * SL;
  const long long CHS = DF ? SL : 1, JS = DF ? 1 : 3LL * D;
  const long long cch = (long long)(h * HD + c) * CHS;
  const int my_slot = my == 0 ? sl0 : sl1;
  const bool my_ok = row_ok(my);
  if (my_ok) {
    const unsigned short* win = reinterpret_cast<const unsigned short*>(a.conv_state) + (long long)my_slot * slot_elems + cch;
#pragma unroll
    for (int kind = 0; kind < 3; ++kind)
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int j = i + SL - 3;  // window slot of sequence position i
        if (j >= 0) xin[kind][i] = win[(long long)kind * D * CHS + j * JS];
      }
  }
  // Row t's quarter q goes into buffer `buf` (bf16: the row's own; fp32: the one buffer)
  // on mbarrier t * 4 + q; thread 0 keeps the mask of the barriers it armed.
  unsigned armed = 0;
  auto issue_quarter = [&](int t, int q, int buf) {
    const unsigned char* src = static_cast<const unsigned char*>(a.state_pool) +
                               ((long long)(t == 0 ? sl0 : sl1) * a.heads + h) * SB::BYTES;
    const uint32_t bar = smem_u32(&mbar[t * QUARTERS + q]);
    mbar_expect_tx(bar, SB::QBYTES);
    bulk_load(smem_u32(smem + S::state + buf * SB::BYTES + q * SB::QBYTES), src + q * SB::QBYTES, SB::QBYTES, bar);
    if constexpr (!BS) armed |= 1u << (t * QUARTERS + q);  // bf16: every good row's copies go out at once
  };
  // fp32: the second row's halves follow the first row's passes, unless the first row
  // has none (padding or a bad slot), in which case they go out now
  const bool row1_later = !BS && row_ok(0) && row_ok(1);
  if (tid == 0) {
#pragma unroll
    for (int q = 0; q < 2 * QUARTERS; ++q) mbar_init(smem_u32(&mbar[q]), 1);
    fence_mbar_init();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (!row_ok(t) || (t == 1 && row1_later)) continue;
#pragma unroll
      for (int q = 0; q < QUARTERS; ++q) issue_quarter(t, q, BS ? t : 0);
    }
    ctl[0] = 0;
  }
  if (tid == 0) slot_s[0] = sl0;
  if (tid == 1) slot_s[1] = sl1;
  fa_b[tid] = fa_v;  // [row][channel] = [tid >> 7][tid & 127]
  gsig_s[tid] = __float2half_rn(sigmoid_fast(bf_bits(gate_v)));
  {
    const float f = bf_bits(fa_v);
    const float sq = warp_sum(f * f);
    if (lane == 0) fnp[my * 4 + c / 32] = sq;
  }
  if (tid < 2) beta_s[tid] = sigmoid_fast(beta_logit);
#pragma unroll
  for (int kind = 0; kind < 3; ++kind) {
    cv[kind].sp[0] = xin[kind][0] | ((unsigned)xin[kind][1] << 16);
    cv[kind].sp[1] = xin[kind][2] | ((unsigned)xin[kind][3] << 16);
  }
  __syncthreads();  // barriers initialised, f_a, its squares and the slots staged

  // ---- causal conv: q, k and v of the thread's channel for its row ---------------------
#pragma unroll
  for (int kind = 0; kind < 3; ++kind) {
    const ConvLane<1>& q = cv[kind];
    float run;
    const float y = conv_dot<0>(q, run);
    const float sy = y * sigmoid_fast(y);  // SiLU; error bound as in the one-row kernel
    float yb;
    if (!bf16_rounding_uncertain(sy, 2.0f * (1.21f * U32 * run + (2.5f * U32 * fabsf(y) + 0x1p-20f) * fabsf(sy))))
      yb = bf_round(sy);
    else
      yb = silu_bf16_exact(bf_bits(q.bb), q.wp[0], q.wp[1], q.sp[0], q.sp[1]);
    if (kind == 0) qh[my * HD + c] = yb;
    else if (kind == 1) kh[my * HD + c] = yb;
    else vv[my * HD + c] = __float2bfloat16_rn(yb);
  }
  // ---- z = f_b . f_a for both rows (even lanes row 0, odd lanes row 1), gate, e^g ------
  {
    const float expA = expf(a_log);
    const uint4* f0 = reinterpret_cast<const uint4*>(fa_b);
    const uint4* f1 = reinterpret_cast<const uint4*>(fa_b + HD);
    float p0[4], p1[4];
    z_partials(fbw, f0[lane & 7], f0[8 + (lane & 7)], p0);
    z_partials(fbw, f1[lane & 7], f1[8 + (lane & 7)], p1);
    float z = z_reduce(p0, lane);
    const float z1 = z_reduce(p1, lane);
    const int tt = lane & 1;
    if (tt) z = z1;
    const float4 np = *reinterpret_cast<const float4*>(fnp + tt * 4);
    const float fnorm = sqrt_fast((np.x + np.y) + (np.z + np.w)) * (1.0f + 0x1p-12f);
    const float bound = 12.0f * U32 * (1.0f + 0x1p-10f) * fbn * fnorm;
    const bool unsure = bf16_rounding_uncertain(z, bound);
    unsigned redo = __ballot_sync(0xffffffffu, unsure);
    z = bf_round(z);
    const int g8 = lane & 24;
    while (redo) {
      const unsigned mine = (redo >> g8) & 0xffu;
      const int li = g8 + (mine ? __ffs(mine) - 1 : 0);
      redo &= ~__ballot_sync(0xffffffffu, mine != 0 && lane == li);
      const uint4* fr = reinterpret_cast<const uint4*>(fa_b + (li & 1) * HD);
      uint4 w0, w1;
      fb_row(fbw, (li >> 1) & 3, w0, w1);
      const float ex = z_exact(w0, w1, fr[lane & 7], fr[8 + (lane & 7)]);
      if (mine != 0 && lane == li) z = ex;
    }
    const float x = z + dtc;
    const float g = (a.gate_mode == KDA_GATE_SOFTPLUS) ? fmaxf(-expA * softplus_fast(x), a.lb)
                                                      : a.lb * sigmoid_fast(expA * x);
    eg[tt * HD + zc] = __expf(g);
  }
  __syncthreads();  // raw q, k, v and e^g of both rows written

  // ---- l2norm of q and k, k^.q^: warp t on row t ---------------------------------------
  if (warp < 2) {
    const int t = warp;
    float4 q = *reinterpret_cast<float4*>(qh + t * HD + lane * 4);
    float4 k = *reinterpret_cast<float4*>(kh + t * HD + lane * 4);
    const float sq = warp_sum(q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
    const float sk = warp_sum(k.x * k.x + k.y * k.y + k.z * k.z + k.w * k.w);
    const float sqk = warp_sum(q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w);
    const float rq = rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
    const float fq = rq * a.q_scale;
    q.x *= fq; q.y *= fq; q.z *= fq; q.w *= fq;
    k.x *= rk; k.y *= rk; k.z *= rk; k.w *= rk;
    *reinterpret_cast<float4*>(qh + t * HD + lane * 4) = q;
    *reinterpret_cast<float4*>(kh + t * HD + lane * 4) = k;
    if (lane == 0) kq_s[t] = sqk * fq * rk;
  }
  __syncthreads();
  // the new window of the thread's row: sequence positions 1..3
  if (my_ok) {
    unsigned short* conv16 = reinterpret_cast<unsigned short*>(a.conv_state);
#pragma unroll
    for (int kind = 0; kind < 3; ++kind) {
      const long long cb = (long long)my_slot * slot_elems + cch + (long long)kind * D * CHS + (long long)(SL - 4) * JS;
#pragma unroll
      for (int p = 1; p <= 3; ++p)
        if (p + SL >= 4) conv16[cb + p * JS] = cv[kind].get(p);
    }
  }

  // ---- recurrence: each row's state in two passes (as the one-row kernel) -------------
  const int hs = lane >> 4, kl = lane & 15;
  const int rbase = warp * 2 + hs;
  const bool b3 = (kl & 8) != 0, b2 = (kl & 4) != 0, b1 = (kl & 2) != 0;
  const int rsel = (b2 ? 2 : 0) + (b1 ? 1 : 0);
  bool timed_out = false;
  bool row1_live = true;  // fp32: the first row's passes put the second row's halves in flight
#pragma unroll 1
  for (int t = 0; t < 2; ++t) {
    if (!row_ok(t) || (t == 1 && !row1_live)) continue;  // uniform across the CTA
    unsigned short* st_t = stb + (BS ? t : 0) * STATE_FLOATS;
    float* stf = st;
    unsigned char* gdst_t = static_cast<unsigned char*>(a.state_pool) + ((long long)(t == 0 ? sl0 : sl1) * a.heads + h) * SB::BYTES;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&mbar[t * QUARTERS + 2 * pass]), 0) &&
                                                  mbar_wait_bounded(smem_u32(&mbar[t * QUARTERS + 2 * pass + 1]), 0));
      if (!ok) timed_out = true;
      // the update of the pass's four rows from the state values in sv
      auto update = [&](float2 (&sv)[4][4]) {
        const int vq = pass * 64 + (rsel >> 1) * 32 + (rsel & 1) * 16 + rbase;
        float2 kv[4], dk2[4], dq2[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) dk2[r] = dq2[r] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int k0 = t * HD + m * 64 + kl * 4;
          const float4 e = *reinterpret_cast<const float4*>(eg + k0);
          const float4 qv = *reinterpret_cast<const float4*>(qh + k0);
          const float4 k4 = *reinterpret_cast<const float4*>(kh + k0);
          const float2 e0 = make_float2(e.x, e.y), e1 = make_float2(e.z, e.w);
          const float2 q0 = make_float2(qv.x, qv.y), q1 = make_float2(qv.z, qv.w);
          kv[2 * m] = make_float2(k4.x, k4.y);
          kv[2 * m + 1] = make_float2(k4.z, k4.w);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            sv[r][2 * m] = mul2(sv[r][2 * m], e0);
            sv[r][2 * m + 1] = mul2(sv[r][2 * m + 1], e1);
            dk2[r] = fma2(sv[r][2 * m], kv[2 * m], dk2[r]);
            dk2[r] = fma2(sv[r][2 * m + 1], kv[2 * m + 1], dk2[r]);
            dq2[r] = fma2(sv[r][2 * m], q0, dq2[r]);
            dq2[r] = fma2(sv[r][2 * m + 1], q1, dq2[r]);
          }
        }
        float v8[8];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          v8[r] = dk2[r].x + dk2[r].y;
          v8[4 + r] = dq2[r].x + dq2[r].y;
        }
        float w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float keep = b3 ? v8[4 + i] : v8[i], send = b3 ? v8[i] : v8[4 + i];
          w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        float w2[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float keep = b2 ? w4[2 + i] : w4[i], send = b2 ? w4[i] : w4[2 + i];
          w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        float rv = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
        rv += __shfl_xor_sync(0xffffffffu, rv, 1);
        const float bt = beta_s[t];
        const float bu_own = bt * (bf(vv[t * HD + vq]) - rv);
        const int src = lane & 16;
        float bu[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) bu[r] = __shfl_sync(0xffffffffu, bu_own, src | (2 * r));
        if (b3 && (kl & 1) == 0) {
          const float bur = b2 ? (b1 ? bu[3] : bu[2]) : (b1 ? bu[1] : bu[0]);
          ob[t * HD + vq] = __float2bfloat16_rn(fmaf(bur, kq_s[t], rv));
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int row = pass * 64 + (r >> 1) * 32 + (r & 1) * 16 + rbase;
          const float2 bu2 = make_float2(bu[r], bu[r]);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            sv[r][2 * m] = fma2(bu2, kv[2 * m], sv[r][2 * m]);
            sv[r][2 * m + 1] = fma2(bu2, kv[2 * m + 1], sv[r][2 * m + 1]);
            if constexpr (BS) {
              const uint2 w = make_uint2(pack_bf16x2(sv[r][2 * m].x, sv[r][2 * m].y),
                                         pack_bf16x2(sv[r][2 * m + 1].x, sv[r][2 * m + 1].y));
              store_streaming_u2(gdst_t + ((long long)row * HD + m * 64 + kl * 4) * 2, w);
            } else {
              store_streaming(reinterpret_cast<float*>(gdst_t + ((long long)row * HD + m * 64 + kl * 4) * 4),
                              make_float4(sv[r][2 * m].x, sv[r][2 * m].y, sv[r][2 * m + 1].x, sv[r][2 * m + 1].y));
            }
          }
        }
      };
      if constexpr (BS) {
        if (ok) {
          float2 sv[4][4];
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const int row = pass * 64 + (r >> 1) * 32 + (r & 1) * 16 + rbase;
              const uint2 x = *reinterpret_cast<const uint2*>(st_t + row * HD + m * 64 + kl * 4);
              sv[r][2 * m] = make_float2(bf_lo(x.x), bf_hi(x.x));
              sv[r][2 * m + 1] = make_float2(bf_lo(x.y), bf_hi(x.y));
            }
          update(sv);
        }
      } else {
        float2 sv[4][4];
        if (ok) {
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const int row = pass * 64 + (r >> 1) * 32 + (r & 1) * 16 + rbase;
              const float4 x = *reinterpret_cast<const float4*>(stf + row * HD + m * 64 + kl * 4);
              sv[r][2 * m] = make_float2(x.x, x.y);
              sv[r][2 * m + 1] = make_float2(x.z, x.w);
            }
        }
        if (t == 0 && row1_later) {  // uniform: this half of the buffer is free once every warp holds its rows
          if (!ok && lane == 0) ctl[0] = 1;
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // these reads before the copy's writes
          __syncthreads();
          // ctl[0] only goes from 0 to 1, and after this barrier only a warp that has given up
          // on a wait of the second row writes it: a warp that reads it late skips that row,
          // which a timeout leaves undefined anyway, and no barrier depends on the choice
          row1_live = ctl[0] == 0;
          if (tid == 0 && row1_live) {
            issue_quarter(1, 2 * pass, 0);
            issue_quarter(1, 2 * pass + 1, 0);
          }
        }
        if (ok) update(sv);
      }
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const float4 onw = *reinterpret_cast<const float4*>(a.o_norm + lane * 4);
  if (timed_out && lane == 0) {
    ctl[0] = 1;
    atomicOr(a.err, KDA_ERR_TIMEOUT);
  }
  __syncthreads();
  if (ctl[0] != 0) {
    if (tid == 0) {
      for (int q = 0; q < 2 * QUARTERS; ++q)
        if (BS ? row_ok(q / QUARTERS) : (armed & (1u << q)) != 0) (void)mbar_wait_bounded(smem_u32(&mbar[q]), 0);
    }
    return;
  }
  // ---- gated RMSNorm: warp t on row t ---------------------------------------------------
  if (warp < 2 && row_ok(warp)) {
    const int t = warp;
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = bf(ob[t * HD + lane * 4 + e]);
    const float ss = warp_sum(o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3]);
    const float rstd = rsqrtf(ss * (1.0f / HD) + a.eps);
    const float wn[4] = {onw.x, onw.y, onw.z, onw.w};
    __align__(8) __nv_bfloat16 y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      y[e] = __float2bfloat16_rn(o[e] * rstd * wn[e] * __half2float(gsig_s[t * HD + lane * 4 + e]));
    *reinterpret_cast<uint2*>(a.out + (row0 + t) * D + h * HD + lane * 4) = *reinterpret_cast<uint2*>(y);
  }
}

// [3D, 1, W] -> [3D] of 4 taps right-aligned (zeros in front when W < 4),
// two bf16 a word: one 8-byte load gives a channel all its taps (the
// PreparedKda page re-lays the weight out once, in decode_conv_weight).
__global__ void pack_conv_w(const unsigned short* in, uint2* out, long long channels, int W) {
  const long long ch = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (ch >= channels) return;
  unsigned short t[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = k - (4 - W);
    t[k] = (j >= 0) ? in[ch * W + j] : (unsigned short)0;
  }
  out[ch] = make_uint2(t[0] | ((unsigned)t[1] << 16), t[2] | ((unsigned)t[3] << 16));
}

#ifdef KDA_DEBUG
// Debug builds only: a step whose rows write the same slot twice is undefined;
// flag it (KDA_ERR_DUPLICATE).  Row i (of a request that is not padding)
// writes slots[i]; each is compared with every later one -- quadratic, which
// a debug build can afford, and it needs no memory beyond the error word.
__global__ void debug_duplicate_slots(const int* slots, long long rows, int L, long long pool, unsigned* err) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < rows; i += (long long)gridDim.x * blockDim.x) {
    const int si = slots[i];
    if (si < 0 || si >= pool || slots[(i / L) * L] == -1) continue;
    for (long long j = i + 1; j < rows; ++j)
      if (slots[j] == si && slots[(j / L) * L] != -1) {
        atomicOr(err, KDA_ERR_DUPLICATE);
        break;
      }
  }
}
#endif

// Euclidean norm of each 128-wide bf16 row, in fp64, rounded up to fp32.
__global__ void row_norms(const __nv_bfloat16* m, float* norms, int rows) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows) return;
  double ss = 0.0;
  for (int j = 0; j < HD; ++j) {
    const double v = (double)__bfloat162float(m[(long long)i * HD + j]);
    ss = fma(v, v, ss);
  }
  norms[i] = __double2float_ru(__dsqrt_ru(ss));
}

template <int L>
cudaError_t set_smem_attr() {
  const cudaError_t e[6] = {
      cudaFuncSetAttribute(kda_step_kernel<L, false, true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Smem<L, false>::bytes),
      cudaFuncSetAttribute(kda_step_kernel<L, true, true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Smem<L, true>::bytes),
      cudaFuncSetAttribute(kda_step_kernel<L, false, false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Smem<L, false>::bytes),
      cudaFuncSetAttribute(kda_step_kernel<L, true, false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Smem<L, true>::bytes),
      cudaFuncSetAttribute(kda_step_kernel<L, false, true, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Smem<L, false>::bytes),
      cudaFuncSetAttribute(kda_step_kernel<L, true, true, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Smem<L, true>::bytes)};
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

cudaError_t set_all_smem_attrs() {
  cudaError_t e = cudaSuccess;
  const cudaError_t d[4] = {
      cudaFuncSetAttribute(kda_decode_pair_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SmemPair<true>::bytes),
      cudaFuncSetAttribute(kda_decode_pair_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SmemPair<true>::bytes),
      cudaFuncSetAttribute(kda_decode_pair_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SmemPair<false>::bytes),
      cudaFuncSetAttribute(kda_decode_pair_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SmemPair<false>::bytes)};
  for (cudaError_t x : d)
    if (x != cudaSuccess) e = x;
  cudaError_t r[KDA_MAX_TOKENS] = {set_smem_attr<1>(), set_smem_attr<2>(), set_smem_attr<3>(), set_smem_attr<4>(),
                                   set_smem_attr<5>(), set_smem_attr<6>(), set_smem_attr<7>(), set_smem_attr<8>()};
  for (int i = 0; i < KDA_MAX_TOKENS; ++i)
    if (r[i] != cudaSuccess) e = r[i];
  return e;
}

template <int L>
cudaError_t launch(const StepArgs& a, long long ctas, cudaStream_t stream, bool bf16_state, bool pdl, int vs) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ctas * vs), 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = bf16_state ? Smem<L, true>::bytes : Smem<L, false>::bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (vs == 2) {  // the two CTAs of a (request, head) as one cluster
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the previous kernel ends
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e;
  if (vs == 2)  // built for the window-first conv layout only
    e = bf16_state ? cudaLaunchKernelEx(&cfg, kda_step_kernel<L, true, true, 2>, a)
                   : cudaLaunchKernelEx(&cfg, kda_step_kernel<L, false, true, 2>, a);
  else if (a.conv_dim_first)
    e = bf16_state ? cudaLaunchKernelEx(&cfg, kda_step_kernel<L, true, true, 1>, a)
                   : cudaLaunchKernelEx(&cfg, kda_step_kernel<L, false, true, 1>, a);
  else
    e = bf16_state ? cudaLaunchKernelEx(&cfg, kda_step_kernel<L, true, false, 1>, a)
                   : cudaLaunchKernelEx(&cfg, kda_step_kernel<L, false, false, 1>, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Decode with a bf16 state pool: two rows of one head a CTA.
cudaError_t launch_decode_pair(const StepArgs& a, long long rows, cudaStream_t stream, bool pdl, bool bs) {
  const long long ctas = (rows + 1) / 2 * a.heads;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = bs ? SmemPair<true>::bytes : SmemPair<false>::bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the previous kernel ends
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (bs)
    e = a.conv_dim_first ? cudaLaunchKernelEx(&cfg, kda_decode_pair_kernel<true, true>, a, (int)rows)
                         : cudaLaunchKernelEx(&cfg, kda_decode_pair_kernel<true, false>, a, (int)rows);
  else
    e = a.conv_dim_first ? cudaLaunchKernelEx(&cfg, kda_decode_pair_kernel<false, true>, a, (int)rows)
                         : cudaLaunchKernelEx(&cfg, kda_decode_pair_kernel<false, false>, a, (int)rows);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int L>
const void* kernel_fn() {
  return reinterpret_cast<const void*>(kda_step_kernel<L, false, true, 1>);
}

bool aligned(const void* p, unsigned n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

}  // namespace

struct kda_handle {
  int device;
  int sms;  // multiprocessors of the device
  int heads, W;
  uint2* conv_w;
  __nv_bfloat16* bias;
  __nv_bfloat16* f_b;
  float* fb_norm;
  float* A_log;
  float* dt_bias;
  float* o_norm;
  unsigned* err;
  float lb, eps;
  int gate_mode;
  int state_dtype;  // KDA_STATE_F32 or KDA_STATE_BF16
  int v_split;      // 1 or 2 CTAs a (request, head)
};

extern "C" {

const char* kda_strerror(int code) {
  switch (code) {
    case KDA_OK: return "ok";
    case KDA_EINVAL: return "invalid argument";
    case KDA_ECUDA: return "CUDA error";
    default: return "unknown error code";
  }
}

void kda_destroy(kda_handle* h) {
  if (h == nullptr) return;
  cudaDeviceSynchronize();
  cudaFree(h->conv_w);
  cudaFree(h->bias);
  cudaFree(h->f_b);
  cudaFree(h->fb_norm);
  cudaFree(h->A_log);
  cudaFree(h->dt_bias);
  cudaFree(h->o_norm);
  cudaFree(h->err);
  delete h;
}

int kda_prepare(int heads, int conv_width, const void* conv_w, const void* bias, const void* f_b,
                const float* A_log, const float* dt_bias, const float* o_norm, float gate_lower_bound,
                float eps, kda_handle** out) {
  if (out == nullptr) return KDA_EINVAL;
  *out = nullptr;
  if (heads < 1 || conv_width < 2 || conv_width > 4 || !(eps > 0.0f)) return KDA_EINVAL;
  if (!conv_w || !f_b || !A_log || !dt_bias || !o_norm) return KDA_EINVAL;
  if (!aligned(conv_w, 2) || !aligned(f_b, 8) || !aligned(A_log, 4) || !aligned(dt_bias, 4) ||
      !aligned(o_norm, 4) || (bias && !aligned(bias, 2)))
    return KDA_EINVAL;
  const long long D = (long long)HD * heads;
  kda_handle* h = new kda_handle();
  h->heads = heads;
  h->W = conv_width;
  h->lb = gate_lower_bound;
  h->gate_mode = KDA_GATE_SIGMOID;
  h->state_dtype = KDA_STATE_F32;
  h->v_split = 1;
  h->eps = eps;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device);
  const size_t conv_bytes = sizeof(uint2) * 3 * D;
  if (e == cudaSuccess) e = cudaMalloc(&h->conv_w, conv_bytes);
  if (e == cudaSuccess && bias) e = cudaMalloc(&h->bias, sizeof(__nv_bfloat16) * 3 * D);
  if (e == cudaSuccess) e = cudaMalloc(&h->f_b, sizeof(__nv_bfloat16) * D * HD);
  if (e == cudaSuccess) e = cudaMalloc(&h->fb_norm, sizeof(float) * D);
  if (e == cudaSuccess) e = cudaMalloc(&h->A_log, sizeof(float) * heads);
  if (e == cudaSuccess) e = cudaMalloc(&h->dt_bias, sizeof(float) * D);
  if (e == cudaSuccess) e = cudaMalloc(&h->o_norm, sizeof(float) * HD);
  if (e == cudaSuccess) e = cudaMalloc(&h->err, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof(unsigned));
  if (e == cudaSuccess && bias) e = cudaMemcpy(h->bias, bias, sizeof(__nv_bfloat16) * 3 * D, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->f_b, f_b, sizeof(__nv_bfloat16) * D * HD, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->A_log, A_log, sizeof(float) * heads, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->dt_bias, dt_bias, sizeof(float) * D, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(h->o_norm, o_norm, sizeof(float) * HD, cudaMemcpyDeviceToDevice);
  if (e == cudaSuccess) {
    pack_conv_w<<<(unsigned)((3 * D + 255) / 256), 256>>>(static_cast<const unsigned short*>(conv_w), h->conv_w,
                                                          3 * D, conv_width);
    e = cudaGetLastError();
  }

  if (e == cudaSuccess) {
    row_norms<<<(unsigned)((D + 255) / 256), 256>>>(h->f_b, h->fb_norm, (int)D);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = set_all_smem_attrs();
  if (e != cudaSuccess) {
    kda_destroy(h);
    return KDA_ECUDA;
  }
  *out = h;
  return KDA_OK;
}

namespace {
int step_enqueue(kda_handle* h, const void* projected, long long rows, long long pitch, void* conv_state,
                 int conv_dim_first, float* state_pool, long long pool_slots, const int* slots, int L,
                 const int* accepted, void* out, void* cuda_stream, bool pdl) {
  if (h == nullptr) return KDA_EINVAL;
  if (L < 1 || L > KDA_MAX_TOKENS || rows < 0 || rows % L != 0 || pool_slots < 0) return KDA_EINVAL;
  const long long D = (long long)HD * h->heads;
  if (pitch < 4 * D + HD + h->heads) return KDA_EINVAL;
  if (rows == 0) return KDA_OK;
  if (L > 1 && accepted == nullptr) return KDA_EINVAL;
  if (!projected || !conv_state || !state_pool || !slots || !out) return KDA_EINVAL;
  if (!aligned(projected, 2) || !aligned(conv_state, 2) || !aligned(state_pool, 16) || !aligned(slots, 4) ||
      !aligned(out, 8) || (accepted && !aligned(accepted, 4)))
    return KDA_EINVAL;
  if (pool_slots > 0x7fffffffLL || rows > 0x7fffffffLL) return KDA_EINVAL;

  StepArgs a;
  a.projected = static_cast<const __nv_bfloat16*>(projected);
  a.pitch = pitch;
  a.conv_state = static_cast<__nv_bfloat16*>(conv_state);
  a.state_pool = state_pool;
  a.pool = pool_slots;
  a.slots = slots;
  a.accepted = accepted;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.conv_w = h->conv_w;
  a.bias = h->bias;
  a.f_b = h->f_b;
  a.fb_norm = h->fb_norm;
  a.A_log = h->A_log;
  a.dt_bias = h->dt_bias;
  a.o_norm = h->o_norm;
  a.err = h->err;
  a.lb = h->lb;
  a.gate_mode = h->gate_mode;
  a.eps = h->eps;
  a.q_scale = 0.08838834764831845f;  // 128^-0.5
  a.heads = h->heads;
  a.D = (int)D;
  a.W = h->W;
  a.conv_dim_first = conv_dim_first ? 1 : 0;

  const long long ctas = (rows / L) * h->heads;
  if (ctas > 0x7fffffffLL) return KDA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const bool bs = h->state_dtype == KDA_STATE_BF16;
#ifdef KDA_DEBUG
  debug_duplicate_slots<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(slots, rows, L, pool_slots, h->err);
  if (cudaGetLastError() != cudaSuccess) return KDA_ECUDA;
#endif
  // One CTA a (request, head) unless the handle asks for two (measured slower on every
  // workload: each half repeats the prologue, and the doubled grid needs more waves).
  int vs = h->v_split;
  if (!a.conv_dim_first) vs = 1;  // the split is built for the window-first conv layout
  if (vs * ctas > 0x7fffffffLL) return KDA_EINVAL;
  cudaError_t e;
  if (L == 1 && vs == 1 && rows >= 2) {  // decode: two rows a CTA
    e = launch_decode_pair(a, rows, s, pdl, bs);
    return e == cudaSuccess ? KDA_OK : KDA_ECUDA;
  }
  switch (L) {
    case 1: e = launch<1>(a, ctas, s, bs, pdl, vs); break;
    case 2: e = launch<2>(a, ctas, s, bs, pdl, vs); break;
    case 3: e = launch<3>(a, ctas, s, bs, pdl, vs); break;
    case 4: e = launch<4>(a, ctas, s, bs, pdl, vs); break;
    case 5: e = launch<5>(a, ctas, s, bs, pdl, vs); break;
    case 6: e = launch<6>(a, ctas, s, bs, pdl, vs); break;
    case 7: e = launch<7>(a, ctas, s, bs, pdl, vs); break;
    default: e = launch<8>(a, ctas, s, bs, pdl, vs); break;
  }
  return e == cudaSuccess ? KDA_OK : KDA_ECUDA;
}
}  // namespace

int kda_step(kda_handle* h, const void* projected, long long rows, long long pitch, void* conv_state,
             int conv_dim_first, float* state_pool, long long pool_slots, const int* slots, int L,
             const int* accepted, void* out, void* cuda_stream) {
  return step_enqueue(h, projected, rows, pitch, conv_state, conv_dim_first, state_pool, pool_slots, slots, L,
                      accepted, out, cuda_stream, false);
}

struct kda_plan {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

int kda_plan_create(kda_handle* h, const void* projected, long long rows, long long pitch, void* conv_state,
                    int conv_dim_first, float* state_pool, long long pool_slots, const int* slots, int L,
                    const int* accepted, void* out, kda_plan** plan) {
  if (plan == nullptr) return KDA_EINVAL;
  *plan = nullptr;
  if (h == nullptr) return KDA_EINVAL;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return KDA_ECUDA;
  cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  int rc = KDA_ECUDA;
  cudaGraph_t g = nullptr;
  if (e == cudaSuccess) {
    rc = kda_step(h, projected, rows, pitch, conv_state, conv_dim_first, state_pool, pool_slots, slots, L, accepted,
                  out, s);
    e = cudaStreamEndCapture(s, &g);  // always ends the capture, whatever kda_step returned
  }
  cudaStreamDestroy(s);
  if (rc != KDA_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return rc != KDA_OK ? rc : KDA_ECUDA;
  }
  cudaGraphExec_t x = nullptr;
  if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return KDA_ECUDA;
  }
  *plan = new kda_plan{g, x};
  return KDA_OK;
}

int kda_layer_plan_create(kda_handle* h, const void* x, long long rows, long long ldx, long long hidden,
                          const void* w_in, void* projected, long long pitch, void* conv_state, int conv_dim_first,
                          float* state_pool, long long pool_slots, const int* slots, int L, const int* accepted,
                          void* core_out, const void* w_o, void* y, long long ldy, int pdl, kda_plan** plan) {
  if (plan == nullptr) return KDA_EINVAL;
  *plan = nullptr;
  if (h == nullptr || rows < 1) return KDA_EINVAL;
  const long long D = (long long)HD * h->heads;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return KDA_ECUDA;
  cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  int rc = KDA_ECUDA;
  cudaGraph_t g = nullptr;
  if (e == cudaSuccess) {
    // in_proj -> projected [rows, pitch]; the core -> core_out [rows, D]; o_proj -> y [rows, hidden]
    rc = kda_linear_enqueue(x, rows, ldx, w_in, pitch, hidden, projected, pitch, s, false);
    if (rc == KDA_OK)
      rc = step_enqueue(h, projected, rows, pitch, conv_state, conv_dim_first, state_pool, pool_slots, slots, L,
                        accepted, core_out, s, (pdl & KDA_PDL_STEP) != 0);
    if (rc == KDA_OK) rc = kda_linear_enqueue(core_out, rows, D, w_o, hidden, D, y, ldy, s, (pdl & KDA_PDL_O_PROJ) != 0);
    e = cudaStreamEndCapture(s, &g);  // always ends the capture, whatever the enqueues returned
  }
  cudaStreamDestroy(s);
  if (rc != KDA_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return rc != KDA_OK ? rc : KDA_ECUDA;
  }
  cudaGraphExec_t xg = nullptr;
  if (cudaGraphInstantiate(&xg, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return KDA_ECUDA;
  }
  *plan = new kda_plan{g, xg};
  return KDA_OK;
}

int kda_plan_launch(kda_plan* p, void* cuda_stream) {
  if (p == nullptr) return KDA_EINVAL;
  return cudaGraphLaunch(p->exec, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

void kda_plan_destroy(kda_plan* p) {
  if (p == nullptr) return;
  cudaGraphExecDestroy(p->exec);
  cudaGraphDestroy(p->graph);
  delete p;
}

int kda_set_state_dtype(kda_handle* h, int dtype) {
  if (h == nullptr || (dtype != KDA_STATE_F32 && dtype != KDA_STATE_BF16)) return KDA_EINVAL;
  h->state_dtype = dtype;
  return KDA_OK;
}

int kda_set_v_split(kda_handle* h, int v_split) {
  if (h == nullptr || (v_split != 1 && v_split != 2)) return KDA_EINVAL;
  h->v_split = v_split;
  return KDA_OK;
}

int kda_set_gate_mode(kda_handle* h, int mode) {
  if (h == nullptr || (mode != KDA_GATE_SIGMOID && mode != KDA_GATE_SOFTPLUS)) return KDA_EINVAL;
  h->gate_mode = mode;
  return KDA_OK;
}

int kda_check(kda_handle* h, void* cuda_stream, unsigned* device_flags) {
  if (h == nullptr) return KDA_EINVAL;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  unsigned flags = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&flags, h->err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof(unsigned));
  if (device_flags) *device_flags = flags;
  return e == cudaSuccess ? KDA_OK : KDA_ECUDA;
}

int kda_launch_info(int L, int* threads, int* smem, int* ctas_per_sm) {
  if (L < 1 || L > KDA_MAX_TOKENS) return KDA_EINVAL;
  const void* fn = nullptr;
  int bytes = 0;
  switch (L) {
    case 1: fn = kernel_fn<1>(); bytes = Smem<1>::bytes; break;
    case 2: fn = kernel_fn<2>(); bytes = Smem<2>::bytes; break;
    case 3: fn = kernel_fn<3>(); bytes = Smem<3>::bytes; break;
    case 4: fn = kernel_fn<4>(); bytes = Smem<4>::bytes; break;
    case 5: fn = kernel_fn<5>(); bytes = Smem<5>::bytes; break;
    case 6: fn = kernel_fn<6>(); bytes = Smem<6>::bytes; break;
    case 7: fn = kernel_fn<7>(); bytes = Smem<7>::bytes; break;
    default: fn = kernel_fn<8>(); bytes = Smem<8>::bytes; break;
  }
  if (threads) *threads = THREADS;
  if (smem) *smem = bytes;
  if (ctas_per_sm) {
    cudaError_t e = set_all_smem_attrs();
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, THREADS, bytes);
    if (e != cudaSuccess) return KDA_ECUDA;
  }
  return KDA_OK;
}

}  // extern "C"
