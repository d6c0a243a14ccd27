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
// Design (one launch per step, one CTA per (request, head)):
//   * stage   -- thread 0 validates the request's slots, then issues the whole
//                64 KiB start state of (slot, head) as four 16 KiB bulk async
//                copies (cp.async.bulk, evict-first L2 hint) into shared
//                memory, each completing on its own mbarrier.  The bytes are
//                in flight before any other work starts (the pages' kda_stage
//                idea: inputs that need no hand-off go first).
//   * prologue, overlapping those copies -- warps 0-3: z = f_b . f_a and the
//                lower-bound gate for the head's 128 decay channels; warps
//                4-7: the causal conv of the head's q, k, v channels over the
//                L tokens and the conv-window stores.  Then one warp per token
//                l2-normalises q and k and computes k^.q^ and beta.
//   * recurrence -- per 32-row quarter of the state (rows = v), a group of 8
//                lanes owns one v row (16 k values per lane, kept in registers
//                across the L tokens); S^T k^ and S^T q^ are reduced with 3
//                xor shuffles; each token's state row goes out with streaming
//                128-bit stores into slots[r, t].  o = S'^T q^ + beta u (k^.q^)
//                with S' the decayed state, an exact reassociation of S_new^T q^.
//   * norm   -- one warp per token: gated RMSNorm of the bf16 o over the
//                head's 128 values -> bf16 core_out.
// Every wait is bounded (1 s of %globaltimer); a wait that gives up sets
// KDA_ERR_TIMEOUT and the affected outputs are not written.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace {

constexpr int HD = 128;                       // head dim (k and v)
constexpr int THREADS = 256;                  // 8 warps
constexpr int STATE_FLOATS = HD * HD;         // one (slot, head) state
constexpr int STATE_BYTES = STATE_FLOATS * 4; // 64 KiB
constexpr int QUARTERS = 4;
constexpr int QUARTER_ROWS = HD / QUARTERS;   // 32 v rows
constexpr int QUARTER_BYTES = STATE_BYTES / QUARTERS;
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;

struct StepArgs {
  const __nv_bfloat16* projected;
  long long pitch;
  __nv_bfloat16* conv_state;
  float* state_pool;
  long long pool;
  const int* slots;
  const int* accepted;
  __nv_bfloat16* out;
  const __nv_bfloat16* conv_w;  // prepared [3][W][D]
  const __nv_bfloat16* bias;    // [3D] or null
  const __nv_bfloat16* f_b;     // [D][128]
  const float* A_log;           // [H]
  const float* dt_bias;         // [D]
  const float* o_norm;          // [128]
  unsigned* err;
  float lb, eps, q_scale;
  int heads, D, W, conv_dim_first;
};

// Shared-memory carve-up for L tokens (byte offsets from the dynamic base).
template <int L>
struct Smem {
  static constexpr int state = 0;
  static constexpr int eg = state + STATE_BYTES;      // float [L][128]  e^g
  static constexpr int kh = eg + L * HD * 4;          // float [L][128]  k, then k^
  static constexpr int qh = kh + L * HD * 4;          // float [L][128]  q, then q^
  static constexpr int vv = qh + L * HD * 4;          // bf16  [L][128]  v
  static constexpr int ob = vv + L * HD * 2;          // bf16  [L][128]  f_a, then o
  static constexpr int beta = ob + L * HD * 2;        // float [L]
  static constexpr int kq = beta + 4 * L;             // float [L]       k^.q^
  static constexpr int slot = kq + 4 * L;             // int   [L]
  static constexpr int ctl = slot + 4 * L;            // int   [4]       status, start, timeout
  static constexpr int mbar = (ctl + 16 + 7) / 8 * 8; // u64   [4]
  static constexpr int bytes = mbar + 8 * QUARTERS;
};

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float bf_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
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

// Wait for phase `parity` of an mbarrier, giving up after WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer() - t0 > WAIT_LIMIT_NS) return false;
  }
  return true;
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

__device__ __forceinline__ void store_streaming(float* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

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
  const float lo = __uint_as_float(a & 0xffff0000u);            // v truncated to bf16
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

__device__ __forceinline__ long long conv_index(const StepArgs& a, long long slot, int ch, int j) {
  const int C = 3 * a.D, SL = a.W - 1;
  return a.conv_dim_first ? (slot * C + ch) * SL + j : (slot * SL + j) * C + ch;
}

template <int L>
__global__ void __launch_bounds__(THREADS, (L <= 4 ? 3 : 2)) kda_step_kernel(const StepArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  using S = Smem<L>;
  float* st = reinterpret_cast<float*>(smem + S::state);
  float* eg = reinterpret_cast<float*>(smem + S::eg);
  float* kh = reinterpret_cast<float*>(smem + S::kh);
  float* qh = reinterpret_cast<float*>(smem + S::qh);
  __nv_bfloat16* vv = reinterpret_cast<__nv_bfloat16*>(smem + S::vv);
  __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(smem + S::ob);
  float* beta_s = reinterpret_cast<float*>(smem + S::beta);
  float* kq_s = reinterpret_cast<float*>(smem + S::kq);
  int* slot_s = reinterpret_cast<int*>(smem + S::slot);
  int* ctl = reinterpret_cast<int*>(smem + S::ctl);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S::mbar);

  const int tid = threadIdx.x;
  const int h = blockIdx.x % a.heads;
  const long long r = blockIdx.x / a.heads;
  const long long row0 = r * L;
  const int D = a.D;

  // ---- stage: validate the request, put the start state in flight --------
  if (tid == 0) {
    const int* sl = a.slots + row0;
    int status = 0, start = 0;
    if (sl[0] == -1) {
      status = 1;  // padding request
    } else {
      int acc = 1;
      if (a.accepted != nullptr) {
        acc = a.accepted[r];
        if (acc < 1 || acc > L) {
          status = 2;
          atomicOr(a.err, KDA_ERR_ACCEPTED);
        }
      }
      if (status == 0) {
        bool bad = false;
#pragma unroll
        for (int t = 0; t < L; ++t) {
          const int s = sl[t];
          slot_s[t] = s;
          bad |= (s < 0) || (s >= a.pool);
        }
        if (bad) {
          status = 2;
          atomicOr(a.err, KDA_ERR_SLOT);
        } else {
          start = sl[acc - 1];
        }
      }
    }
    ctl[0] = status;
    ctl[1] = start;
    ctl[2] = 0;
    if (status == 0) {
      const float* src = a.state_pool + ((long long)start * a.heads + h) * STATE_FLOATS;
#pragma unroll
      for (int q = 0; q < QUARTERS; ++q) mbar_init(smem_u32(&mbar[q]), 1);
      fence_mbar_init();
#pragma unroll
      for (int q = 0; q < QUARTERS; ++q) {
        const uint32_t bar = smem_u32(&mbar[q]);
        mbar_expect_tx(bar, QUARTER_BYTES);
        bulk_load(smem_u32(st + q * QUARTER_ROWS * HD), src + q * QUARTER_ROWS * HD, QUARTER_BYTES, bar);
      }
    }
  }
  __syncthreads();
  const int status = ctl[0];
  if (status == 1) {  // padding: zero output rows, no cache traffic
    for (int i = tid; i < L * HD; i += THREADS)
      a.out[(row0 + i / HD) * D + h * HD + (i % HD)] = __float2bfloat16_rn(0.0f);
    return;
  }
  if (status != 0) return;
  const int start = ctl[1];

  // ---- prologue: f_a staging ------------------------------------------------
  for (int i = tid; i < L * HD; i += THREADS)
    ob[i] = a.projected[(row0 + i / HD) * a.pitch + 4 * D + (i % HD)];
  __syncthreads();

  if (tid < HD) {
    // z = f_b . f_a for decay channel c of head h, then the lower-bound gate.
    const int c = tid;
    const uint4* fbrow = reinterpret_cast<const uint4*>(a.f_b + (long long)(h * HD + c) * HD);
    float acc[L], run[L];  // the fp32 dot and the sum of |partial sums| (its error bound / u)
#pragma unroll
    for (int t = 0; t < L; ++t) acc[t] = run[t] = 0.0f;
#pragma unroll 2
    for (int j8 = 0; j8 < HD / 8; ++j8) {
      const uint4 w = __ldg(fbrow + j8);
      const __nv_bfloat16* wb = reinterpret_cast<const __nv_bfloat16*>(&w);
      float wf[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) wf[e] = bf(wb[e]);
#pragma unroll
      for (int t = 0; t < L; ++t) {
        const uint4 fa = *reinterpret_cast<const uint4*>(ob + t * HD + j8 * 8);
        const __nv_bfloat16* fb = reinterpret_cast<const __nv_bfloat16*>(&fa);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          acc[t] = fmaf(wf[e], bf(fb[e]), acc[t]);  // bf16 x bf16 products are exact in fp32
          run[t] += fabsf(acc[t]);
        }
      }
    }
    const float expA = expf(a.A_log[h]);
    const float dtc = a.dt_bias[h * HD + c];
#pragma unroll
    for (int t = 0; t < L; ++t) {
      // |acc - exact| <= u (1 + 2u) sum|partials|; margin x2
      float z;
      if (!bf16_rounding_uncertain(acc[t], 2.0f * U32 * run[t])) {
        z = bf_round(acc[t]);
      } else {
        // compensated (TwoSum) re-summation: s + e carries the exact dot up to
        // an error of order n^2 u^2 sum|p|, then one correctly rounded conversion.
        const __nv_bfloat16* row = a.f_b + (long long)(h * HD + c) * HD;
        float sum = 0.0f, err = 0.0f;
        for (int j = 0; j < HD; ++j) {
          const float p = bf(row[j]) * bf(ob[t * HD + j]);
          const float nsum = sum + p;
          const float bp = nsum - sum;
          err += (sum - (nsum - bp)) + (p - bp);
          sum = nsum;
        }
        z = bf16_round_f64((double)sum + (double)err);
      }
      const float g = a.lb * sigmoidf_(expA * (z + dtc));
      eg[t * HD + c] = expf(g);
    }
  } else {
    // causal depthwise conv of channel i in the head's q, k and v blocks.
    const int i = tid - HD;
    const int SL = a.W - 1;
#pragma unroll 1
    for (int blk = 0; blk < 3; ++blk) {
      const int ch = blk * D + h * HD + i;
      float win[3] = {0.0f, 0.0f, 0.0f}, w[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < 3; ++j)
        if (j < SL) win[j] = bf(a.conv_state[conv_index(a, start, ch, j)]);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < a.W) w[j] = bf(a.conv_w[(long long)(blk * a.W + j) * D + h * HD + i]);
      const float b = a.bias ? bf(a.bias[ch]) : 0.0f;
      float w_cur = 0.0f;  // the tap on the current token, w[SL]
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j == SL) w_cur = w[j];
#pragma unroll
      for (int t = 0; t < L; ++t) {
        const float x = bf(a.projected[(row0 + t) * a.pitch + ch]);
        float y = b, run = 0.0f;  // run: sum of |partial sums|, the fp32 error bound / u
#pragma unroll
        for (int j = 0; j < 3; ++j)
          if (j < SL) {
            y = fmaf(w[j], win[j], y);
            run += fabsf(y);
          }
        y = fmaf(w_cur, x, y);
        run += fabsf(y);
        const float sy = y * sigmoidf_(y);  // SiLU
        // |sy - silu(exact y)| <= 1.1 u (1+2u) run + 2^-21 |sy| (expf within 2 ulp); margin x2
        float yb;
        if (!bf16_rounding_uncertain(sy, 2.0f * (1.1f * U32 * run + 4.0f * U32 * fabsf(sy)))) {
          yb = bf_round(sy);
        } else {
          double yd = (double)b;
#pragma unroll
          for (int j = 0; j < 3; ++j)
            if (j < SL) yd = fma((double)w[j], (double)win[j], yd);
          yd = fma((double)w_cur, (double)x, yd);
          yb = bf16_round_f64(yd / (1.0 + exp(-yd)));
        }
        if (blk == 0) qh[t * HD + i] = yb;
        else if (blk == 1) kh[t * HD + i] = yb;
        else vv[t * HD + i] = __float2bfloat16_rn(yb);
#pragma unroll
        for (int j = 0; j < 3; ++j)
          win[j] = (j + 1 < SL) ? win[j + 1] : (j + 1 == SL ? x : win[j]);
        const long long dst = slot_s[t];
#pragma unroll
        for (int j = 0; j < 3; ++j)
          if (j < SL) a.conv_state[conv_index(a, dst, ch, j)] = __float2bfloat16_rn(win[j]);
      }
    }
  }
  __syncthreads();

  // ---- l2norm of q and k, k^.q^, beta: one warp per token --------------------
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < L) {
    const int t = warp;
    float4 q = *reinterpret_cast<float4*>(qh + t * HD + lane * 4);
    float4 k = *reinterpret_cast<float4*>(kh + t * HD + lane * 4);
    const float sq = warp_sum(q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
    const float sk = warp_sum(k.x * k.x + k.y * k.y + k.z * k.z + k.w * k.w);
    const float qk = warp_sum(q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w);
    const float rq = 1.0f / sqrtf(sq + 1e-6f), rk = 1.0f / sqrtf(sk + 1e-6f);
    const float fq = rq * a.q_scale;
    q.x *= fq; q.y *= fq; q.z *= fq; q.w *= fq;
    k.x *= rk; k.y *= rk; k.z *= rk; k.w *= rk;
    *reinterpret_cast<float4*>(qh + t * HD + lane * 4) = q;
    *reinterpret_cast<float4*>(kh + t * HD + lane * 4) = k;
    if (lane == 0) {
      kq_s[t] = qk * fq * rk;
      beta_s[t] = sigmoidf_(bf(a.projected[(row0 + t) * a.pitch + 4 * D + HD + h]));
    }
  }
  __syncthreads();

  // ---- recurrence: a group of 8 lanes per v row, 16 k values per lane --------
  const int sub = lane >> 3, kl = lane & 7;
  bool any_timeout = false;
#pragma unroll 1
  for (int qtr = 0; qtr < QUARTERS; ++qtr) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&mbar[qtr]), 0));
    if (!ok) {
      any_timeout = true;
      continue;
    }
    const int v = qtr * QUARTER_ROWS + warp * 4 + sub;
    float4 s[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] = *reinterpret_cast<const float4*>(st + v * HD + j * 32 + kl * 4);
#pragma unroll 1
    for (int t = 0; t < L; ++t) {
      float4 kv[4];
      float dk = 0.0f, dq = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k0 = t * HD + j * 32 + kl * 4;
        const float4 e = *reinterpret_cast<const float4*>(eg + k0);
        const float4 qv = *reinterpret_cast<const float4*>(qh + k0);
        kv[j] = *reinterpret_cast<const float4*>(kh + k0);
        s[j].x *= e.x; s[j].y *= e.y; s[j].z *= e.z; s[j].w *= e.w;
        dk = fmaf(s[j].x, kv[j].x, dk); dk = fmaf(s[j].y, kv[j].y, dk);
        dk = fmaf(s[j].z, kv[j].z, dk); dk = fmaf(s[j].w, kv[j].w, dk);
        dq = fmaf(s[j].x, qv.x, dq); dq = fmaf(s[j].y, qv.y, dq);
        dq = fmaf(s[j].z, qv.z, dq); dq = fmaf(s[j].w, qv.w, dq);
      }
#pragma unroll
      for (int m = 1; m <= 4; m <<= 1) {
        dk += __shfl_xor_sync(0xffffffffu, dk, m);
        dq += __shfl_xor_sync(0xffffffffu, dq, m);
      }
      const float u = bf(vv[t * HD + v]) - dk;
      const float bu = beta_s[t] * u;
      const float o = fmaf(bu, kq_s[t], dq);
      float* dst = a.state_pool + (((long long)slot_s[t] * a.heads + h) * HD + v) * HD + kl * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        s[j].x = fmaf(bu, kv[j].x, s[j].x); s[j].y = fmaf(bu, kv[j].y, s[j].y);
        s[j].z = fmaf(bu, kv[j].z, s[j].z); s[j].w = fmaf(bu, kv[j].w, s[j].w);
        store_streaming(dst + j * 32, s[j]);
      }
      if (kl == 0) ob[t * HD + v] = __float2bfloat16_rn(o);
    }
  }
  if (any_timeout) {
    if (lane == 0) {
      ctl[2] = 1;
      atomicOr(a.err, KDA_ERR_TIMEOUT);
    }
  }
  __syncthreads();
  if (ctl[2] != 0) {
    // Give copies still in flight a second bounded chance to land before the
    // shared memory is released; the outputs of this request stay unwritten.
    if (tid == 0)
      for (int q = 0; q < QUARTERS; ++q) (void)mbar_wait_bounded(smem_u32(&mbar[q]), 0);
    return;
  }

  // ---- gated RMSNorm: one warp per token ---------------------------------------
  if (warp < L) {
    const int t = warp;
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = bf(ob[t * HD + lane * 4 + e]);
    const float ss = warp_sum(o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3]);
    const float rstd = 1.0f / sqrtf(ss * (1.0f / HD) + a.eps);
    const __nv_bfloat16* gate = a.projected + (row0 + t) * a.pitch + 3 * D + h * HD + lane * 4;
    __align__(8) __nv_bfloat16 y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      y[e] = __float2bfloat16_rn(o[e] * rstd * a.o_norm[lane * 4 + e] * sigmoidf_(bf(gate[e])));
    *reinterpret_cast<uint2*>(a.out + (row0 + t) * D + h * HD + lane * 4) = *reinterpret_cast<uint2*>(y);
  }
}

// [3D, 1, W] -> [3, W, D] (decode_conv_weight on the PreparedKda page).
__global__ void relayout_conv_w(const __nv_bfloat16* in, __nv_bfloat16* out, int D, int W) {
  const long long n = 3LL * D * W;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long ch = i / W;  // source channel in [0, 3D)
    const int j = (int)(i % W);
    const long long blk = ch / D, c = ch % D;
    out[(blk * W + j) * D + c] = in[i];
  }
}

template <int L>
int smem_bytes() {
  return Smem<L>::bytes;
}

template <int L>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(kda_step_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<L>::bytes);
}

template <int L>
cudaError_t launch(const StepArgs& a, long long ctas, cudaStream_t stream) {
  kda_step_kernel<L><<<(unsigned)ctas, THREADS, Smem<L>::bytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t set_all_smem_attrs() {
  cudaError_t e = cudaSuccess;
  cudaError_t r[KDA_MAX_TOKENS] = {set_smem_attr<1>(), set_smem_attr<2>(), set_smem_attr<3>(), set_smem_attr<4>(),
                                   set_smem_attr<5>(), set_smem_attr<6>(), set_smem_attr<7>(), set_smem_attr<8>()};
  for (int i = 0; i < KDA_MAX_TOKENS; ++i)
    if (r[i] != cudaSuccess) e = r[i];
  return e;
}

bool aligned(const void* p, unsigned n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

}  // namespace

struct kda_handle {
  int device;
  int heads, W;
  __nv_bfloat16* conv_w;
  __nv_bfloat16* bias;
  __nv_bfloat16* f_b;
  float* A_log;
  float* dt_bias;
  float* o_norm;
  unsigned* err;
  float lb, eps;
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
  if (!aligned(conv_w, 2) || !aligned(f_b, 2) || !aligned(A_log, 4) || !aligned(dt_bias, 4) ||
      !aligned(o_norm, 4) || (bias && !aligned(bias, 2)))
    return KDA_EINVAL;
  const long long D = (long long)HD * heads;
  kda_handle* h = new kda_handle();
  h->heads = heads;
  h->W = conv_width;
  h->lb = gate_lower_bound;
  h->eps = eps;
  cudaError_t e = cudaGetDevice(&h->device);
  const size_t conv_bytes = sizeof(__nv_bfloat16) * 3 * D * conv_width;
  if (e == cudaSuccess) e = cudaMalloc(&h->conv_w, conv_bytes);
  if (e == cudaSuccess && bias) e = cudaMalloc(&h->bias, sizeof(__nv_bfloat16) * 3 * D);
  if (e == cudaSuccess) e = cudaMalloc(&h->f_b, sizeof(__nv_bfloat16) * D * HD);
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
    relayout_conv_w<<<(unsigned)((3 * D * conv_width + 255) / 256), 256>>>(
        static_cast<const __nv_bfloat16*>(conv_w), h->conv_w, (int)D, conv_width);
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

int kda_step(kda_handle* h, const void* projected, long long rows, long long pitch, void* conv_state,
             int conv_dim_first, float* state_pool, long long pool_slots, const int* slots, int L,
             const int* accepted, void* out, void* cuda_stream) {
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
  const long long ctas = (rows / L) * h->heads;
  if (ctas > 0x7fffffffLL) return KDA_EINVAL;

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
  a.A_log = h->A_log;
  a.dt_bias = h->dt_bias;
  a.o_norm = h->o_norm;
  a.err = h->err;
  a.lb = h->lb;
  a.eps = h->eps;
  a.q_scale = 0.08838834764831845f;  // 128^-0.5
  a.heads = h->heads;
  a.D = (int)D;
  a.W = h->W;
  a.conv_dim_first = conv_dim_first ? 1 : 0;

  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e;
  switch (L) {
    case 1: e = launch<1>(a, ctas, s); break;
    case 2: e = launch<2>(a, ctas, s); break;
    case 3: e = launch<3>(a, ctas, s); break;
    case 4: e = launch<4>(a, ctas, s); break;
    case 5: e = launch<5>(a, ctas, s); break;
    case 6: e = launch<6>(a, ctas, s); break;
    case 7: e = launch<7>(a, ctas, s); break;
    default: e = launch<8>(a, ctas, s); break;
  }
  return e == cudaSuccess ? KDA_OK : KDA_ECUDA;
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
    case 1: fn = (const void*)kda_step_kernel<1>; bytes = smem_bytes<1>(); break;
    case 2: fn = (const void*)kda_step_kernel<2>; bytes = smem_bytes<2>(); break;
    case 3: fn = (const void*)kda_step_kernel<3>; bytes = smem_bytes<3>(); break;
    case 4: fn = (const void*)kda_step_kernel<4>; bytes = smem_bytes<4>(); break;
    case 5: fn = (const void*)kda_step_kernel<5>; bytes = smem_bytes<5>(); break;
    case 6: fn = (const void*)kda_step_kernel<6>; bytes = smem_bytes<6>(); break;
    case 7: fn = (const void*)kda_step_kernel<7>; bytes = smem_bytes<7>(); break;
    default: fn = (const void*)kda_step_kernel<8>; bytes = smem_bytes<8>(); break;
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
