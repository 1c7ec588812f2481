// spec_verify.cu -- batched speculative-sampling verify step for GB300 (sm_103a).
//
// What is computed (per request b, gamma_b drafts, vocabulary V, temperature T):
//   p_i = softmax(t[b][i]/T), q_i = softmax(d[b][i]/T); accept x_i iff
//   u_i < p_i(x_i)/q_i(x_i); k = first rejected position (else gamma_b); one
//   token drawn at k from max(0, p_k - q_k) (or from p_{gamma_b} as the bonus)
//   by the inverse CDF over ascending token id against u[b][G].
//   (disassemble-channel "Speculative Decoding theory", Step 3 and the
//   "modified distribution" section; "Fast Inference from Transformers via
//   Speculative Decoding" explainer, algorithm section; toolsku "LLM
//   speculative decoding optimisation", verify sketch with the bonus token.)
//   Greedy: argmax match (explainer, "Implementation points", greedy note).
//
// One persistent kernel per call.  CTAs claim work items from one atomic
// counter, in a fixed global order:
//   A item  16 KB of one logit row (row statistics).  Per warp: the chunk
//           maximum and the sum of exp2((z - max) log2(e)/T) (sampling), or
//           the argmax (greedy), written as a per-warp partial.
//   R item  8 KB of the target row k and the same 8 KB of the draft row k
//           of one request (sampling only): the fixed-point (2^-39) sum of the
//           residual weights max(0, p_k - q_k) (or of p for the bonus draw).
// The order is request-major: the A items of request b, then the R items of
// request b - L.  The lag L keeps R items behind their request's decision,
// while the rows are still in L2.  The CTA whose A item completes a request
// (atomic arrival count) combines the partials in float64, runs the
// acceptance tests with a warp-ballot first-reject scan, and publishes the
// request's decision; the CTA whose R item completes it locates the chunk that
// holds u*S and scans only that chunk for the token.  A CTA waits for a
// decision only while it holds no unfinished item, so waits always end; every
// wait is also bounded by an iteration limit that sets SV_STATUS_TIMEOUT.
// Counters are reset by their last user, so the workspace stays zeroed.
//
// Numerics: inputs widen exactly to float32.  Exponent arguments use a
// two-term log2(e)/T (hi + lo); exp2 is the SFU's ex2.approx; sums inside a
// warp are float32, sums across warps and chunks float64.  The acceptance
// ratio is formed in float64.  The residual CDF is summed in exact 64-bit
// fixed point, so chunk sums and the final in-chunk scan agree bit for bit.

#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>
#include <float.h>

#include "spec_verify.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVecA = 4;                              // 16-byte vectors per thread per A item
constexpr int kTileBytes = kThreads * kVecA * 16;     // 16 KB of one row per A item
constexpr int kHalfBytes = kTileBytes / 2;            // 8 KB of each row per R item
constexpr int kMaxBatch = 8192;                       // requests per launch (smem prefix)
constexpr unsigned kSpinLimit = 1u << 22;             // bounded waits
constexpr float kFix = 549755813888.0f;               // 2^39: fixed-point scale of probabilities
constexpr float kLog2eHi = 1.44269502162933349609375f;      // float nearest log2(e)
constexpr float kLog2eLo = 1.925963033500011e-08f;          // log2(e) - kLog2eHi

enum { KIND_A = 0, KIND_R = 1, KIND_RWAIT = 2, KIND_EXIT = 3 };
enum { MODE_SAMPLE = 0, MODE_GREEDY = 1 };

// ---------------------------------------------------------------------------
// Workspace
// ---------------------------------------------------------------------------
struct Decision {      // per request, published by the deciding CTA
  int k;               // first rejected position (gamma_b if none)
  int reject;          // 1: residual at k; 0: bonus from target row k = gamma_b
  float mt, md;        // maxima of target row k and draft row k
  float inv_st, rho;   // 1/S_t and S_t/S_d of those rows (float64-derived)
  float c_hi, c_lo;    // log2(e)/T as hi + lo
};

struct Layout {
  size_t status, next_item, exit_count;  // header words
  size_t cnt_a, cnt_r, ready, dec, stats, resid, total;
  int NC, NCR;  // worst-case chunk counts (float32 logits)
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline Layout make_layout(int B, int G, int V) {
  Layout L;
  L.NC = (V + kTileBytes / 4 - 1) / (kTileBytes / 4);
  L.NCR = (V + kHalfBytes / 4 - 1) / (kHalfBytes / 4);
  L.status = 0;
  L.next_item = 64;
  L.exit_count = 128;
  size_t off = 256;
  L.cnt_a = off; off = align256(off + (size_t)B * 4);
  L.cnt_r = off; off = align256(off + (size_t)B * 4);
  L.ready = off; off = align256(off + (size_t)B * 4);
  L.dec = off;   off = align256(off + (size_t)B * sizeof(Decision));
  L.stats = off; off = align256(off + (size_t)B * (2 * G + 1) * L.NC * kWarps * sizeof(float2));
  L.resid = off; off = align256(off + (size_t)B * L.NCR * sizeof(ulonglong2));
  L.total = off;
  return L;
}

struct Params {
  const char* target;
  const char* draft;
  int B, G, V, NC, NCR;       // NC/NCR: chunk counts for this dtype
  int stride_nc, stride_ncr;  // allocated chunk counts (workspace strides)
  const int32_t* tokens;
  const int32_t* gamma;
  const float* uniforms;
  const float* temperature;
  int32_t* out_tokens;
  int32_t* num_accepted;
  double* p_tok;
  double* q_tok;
  unsigned int* status;
  unsigned int* next_item;
  unsigned int* exit_count;
  unsigned int* cnt_a;
  unsigned int* cnt_r;
  unsigned int* ready;
  Decision* dec;
  float2* stats;       // [B][2G+1][stride_nc][kWarps] (m, s) or (m, idx bits)
  ulonglong2* resid;   // [B][stride_ncr] (residual sum, p sum)
};

// Work item, decoded by thread 0 into shared memory.
struct Slot {
  int kind;
  int b;
  int pslot;    // A: partial row slot; R: k
  int c;        // chunk index
  int n;        // valid elements (A: in the tile; R: per row)
  int aligned;  // all row pointers 16-byte aligned
  int reject;   // R
  int pad;
  const char* p0;  // A: tile start; R: target half-tile
  const char* p1;  // R: draft half-tile, or null for the bonus draw
  float mt, md, inv_st, rho, c_hi, c_lo;
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Decision record read through L2 (it was written by another CTA).
__device__ __forceinline__ Decision load_decision(const Decision* p) {
  static_assert(sizeof(Decision) == 32, "Decision is two 16-byte words");
  const uint4* q = reinterpret_cast<const uint4*>(p);
  const uint4 a = __ldcg(q), b = __ldcg(q + 1);
  Decision d;
  d.k = (int)a.x;
  d.reject = (int)a.y;
  d.mt = __uint_as_float(a.z);
  d.md = __uint_as_float(a.w);
  d.inv_st = __uint_as_float(b.x);
  d.rho = __uint_as_float(b.y);
  d.c_hi = __uint_as_float(b.z);
  d.c_lo = __uint_as_float(b.w);
  return d;
}

template <int EB>
__device__ __forceinline__ float load_elem(const char* base, size_t idx) {
  if (EB == 2) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
    return __uint_as_float((uint32_t)h << 16);
  } else {
    return __ldg(reinterpret_cast<const float*>(base) + idx);
  }
}

// element j of a 16-byte vector holding VEC = 16/EB logits
template <int EB>
__device__ __forceinline__ float vec_elem(const uint4& v, int j) {
  const uint32_t w = j < (EB == 2 ? 2 : 1) ? v.x : j < (EB == 2 ? 4 : 2) ? v.y
                   : j < (EB == 2 ? 6 : 3) ? v.z : v.w;
  if (EB == 2) return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  return __uint_as_float(w);
}

__device__ __forceinline__ int clamp_gamma(int g, int G) { return g < 0 ? 0 : (g > G ? G : g); }

struct TempC {
  float hi, lo;  // log2(e)/T = hi + lo, hi rounded toward zero so lo > 0
};

// Two-term log2(e)/T in float arithmetic: hi = RZ(L/T); the FMA gives the
// exact remainder L_hi - hi*T, from which lo follows.  lo is kept >= FLT_MIN
// so that -inf logits give -inf arguments rather than NaN.
__device__ __forceinline__ TempC temp_consts(float T) {
  TempC t;
  t.hi = __fdiv_rz(kLog2eHi, T);
  const float r = __fmaf_rn(-t.hi, T, kLog2eHi);
  t.lo = __fdiv_rn(__fadd_rn(r, kLog2eLo), T);
  if (!(t.lo >= FLT_MIN)) t.lo = FLT_MIN;
  return t;
}

__device__ __forceinline__ float sanitize_temperature(float T, unsigned int& flags) {
  if (!(T > 0.0f) || isinf(T)) {
    flags |= SV_STATUS_BAD_TEMPERATURE;
    return 1.0f;
  }
  return T;
}

__device__ __forceinline__ float sanitize_uniform(float u, unsigned int& flags) {
  if (!(u >= 0.0f && u < 1.0f)) {
    flags |= SV_STATUS_BAD_UNIFORM;
    return 0.0f;
  }
  return u;
}

// (z - m) * log2(e)/T with the two-term constant; explicit round-to-nearest
// intrinsics so every call site computes identical bits.
__device__ __forceinline__ float exp_arg(float z, float m, float hi, float lo) {
  const float d = __fsub_rn(z, m);
  return __fmaf_rn(d, hi, __fmul_rn(d, lo));
}

__device__ __forceinline__ size_t target_row(int b, int i, int G, int V) {
  return ((size_t)b * (size_t)(G + 1) + (size_t)i) * (size_t)V;
}
__device__ __forceinline__ size_t draft_row(int b, int i, int G, int V) {
  return ((size_t)b * (size_t)G + (size_t)i) * (size_t)V;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ void argmax_combine(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_combine(v, i, v2, i2);
  }
}

// Loads NV 16-byte vectors per thread (vector index threadIdx.x + k*kThreads)
// of a tile starting at p with n valid elements into buf[off..off+NV).  The
// fast path is one non-caching 16-byte load per vector; vectors past the end
// or in an unaligned tile are assembled from scalar loads, with -inf filling
// missing elements.
template <int EB, int NV>
__device__ __forceinline__ void load_tile(uint4* buf, const char* p, int n, bool aligned) {
  constexpr int VEC = 16 / EB;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int e0 = ((int)threadIdx.x + k * kThreads) * VEC;
    if (aligned && e0 + VEC <= n) {
      buf[k] = ldg_stream(p + (size_t)e0 * EB);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (EB == 2) {
          const int ea = e0 + 2 * q, eb = ea + 1;
          const uint32_t lo = ea < n ? __ldg(reinterpret_cast<const unsigned short*>(p) + ea) : 0xff80u;
          const uint32_t hi = eb < n ? __ldg(reinterpret_cast<const unsigned short*>(p) + eb) : 0xff80u;
          w[q] = lo | (hi << 16);
        } else {
          const int e = e0 + q;
          w[q] = e < n ? __float_as_uint(__ldg(reinterpret_cast<const float*>(p) + e)) : 0xff800000u;
        }
      }
      buf[k] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

__device__ __forceinline__ void fill_neg_inf(uint4* buf, int nv, int eb) {
  const uint32_t f = eb == 2 ? 0xff80ff80u : 0xff800000u;
  for (int k = 0; k < nv; ++k) buf[k] = make_uint4(f, f, f, f);
}

// ---------------------------------------------------------------------------
// Residual weights (shared by R items and the final in-chunk scan)
// r = max(0, p - q) = (1/S_t) * max(0, e_t - e_d * S_t/S_d), in fixed point.
// ---------------------------------------------------------------------------
struct ResidC {
  float mt, md, inv_st, rho, hi, lo;
  int reject;
};

__device__ __forceinline__ void resid_weights(float zt, float zd, const ResidC& k,
                                              unsigned long long& wr, unsigned long long& wp) {
  const float et = ex2_approx(exp_arg(zt, k.mt, k.hi, k.lo));
  const float pv = __fmul_rn(et, k.inv_st);
  wp = __float2ull_rn(__fmul_rn(pv, kFix));
  if (k.reject) {
    const float ed = ex2_approx(exp_arg(zd, k.md, k.hi, k.lo));
    const float rv = __fmul_rn(fmaxf(__fmaf_rn(-ed, k.rho, et), 0.0f), k.inv_st);
    wr = __float2ull_rn(__fmul_rn(rv, kFix));
  } else {
    wr = wp;
  }
}

// floor(u * S) exactly, for u a float in [0, 1).
__device__ __forceinline__ unsigned long long scaled_target(float u, unsigned long long S) {
  const uint32_t bits = __float_as_uint(u);
  const uint32_t ex = (bits >> 23) & 0xffu;
  const uint32_t frac = bits & 0x7fffffu;
  if (ex == 0 && frac == 0) return 0ull;
  const unsigned long long M = ex ? (frac | 0x800000u) : frac;
  const int shift = ex ? 150 - (int)ex : 149;  // u = M * 2^-shift
  const unsigned __int128 prod = (unsigned __int128)M * (unsigned __int128)S;
  return shift >= 128 ? 0ull : (unsigned long long)(prod >> shift);
}

__device__ __forceinline__ unsigned long long block_exclusive_scan(unsigned long long v,
                                                                   unsigned long long* sh,
                                                                   unsigned long long* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < kWarps ? sh[lane] : 0ull;
    unsigned long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) sh[kWarps + lane] = wi - w;
    if (lane == kWarps - 1) sh[2 * kWarps] = wi;
  }
  __syncthreads();
  const unsigned long long excl = sh[kWarps + warp] + (incl - v);
  *total = sh[2 * kWarps];
  __syncthreads();
  return excl;
}

// ---------------------------------------------------------------------------
// Per-request decision (sampling), run by the whole CTA that completed the
// request's last A item.
// ---------------------------------------------------------------------------
template <int EB>
__device__ __noinline__ void decide_sample(const Params& P, int b) {
  __shared__ float s_m[2 * SV_MAX_GAMMA + 1];
  __shared__ double s_s[2 * SV_MAX_GAMMA + 1];
  const int G = P.G, V = P.V, NC = P.NC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gb = clamp_gamma(P.gamma[b], G);
  unsigned int flags = (P.gamma[b] != gb) ? SV_STATUS_BAD_GAMMA : 0u;
  const float T = sanitize_temperature(P.temperature[b], flags);
  const TempC tc = temp_consts(T);
  const double cd = (double)tc.hi + (double)tc.lo;
  const int nrows = 2 * gb + 1;
  const int nparts = NC * kWarps;

  // Row maximum M and normaliser S = sum_w s_w 2^((m_w - M) c) over the
  // per-warp partials, combined in float64.
  for (int r = warp; r < nrows; r += kWarps) {
    const int slot = r <= gb ? r : (G + 1 + (r - gb - 1));
    const float2* pr = P.stats + ((size_t)b * (2 * G + 1) + slot) * P.stride_nc * kWarps;
    float M = -INFINITY;
    for (int j = lane; j < nparts; j += 32) M = fmaxf(M, __ldcg(&pr[j]).x);
    M = warp_max(M);
    double S = 0.0;
    if (M > -INFINITY) {
      for (int j = lane; j < nparts; j += 32) {
        const float2 ms = __ldcg(&pr[j]);
        if (ms.x > -INFINITY) S += (double)ms.y * (double)ex2_approx(exp_arg(ms.x, M, tc.hi, tc.lo));
      }
    }
    S = warp_sum_d(S);
    if (lane == 0) {
      s_m[r] = M;
      s_s[r] = S;
      if (!isfinite(M) || !(S > 0.0)) flags |= SV_STATUS_NONFINITE_ROW;
    }
  }
  __syncthreads();

  if (warp == 0) {
    const int i = lane;
    bool reject = false;
    double p = NAN, q = NAN;
    int x = 0;
    if (i < gb) {
      x = P.tokens[(size_t)b * G + i];
      if (x < 0 || x >= V) {
        flags |= SV_STATUS_BAD_TOKEN;
        x = x < 0 ? 0 : V - 1;
      }
      const float zt = load_elem<EB>(P.target, target_row(b, i, G, V) + (size_t)x);
      const float zd = load_elem<EB>(P.draft, draft_row(b, i, G, V) + (size_t)x);
      p = exp2(((double)zt - (double)s_m[i]) * cd) / s_s[i];
      q = exp2(((double)zd - (double)s_m[gb + 1 + i]) * cd) / s_s[gb + 1 + i];
      const double u = (double)sanitize_uniform(P.uniforms[(size_t)b * (G + 1) + i], flags);
      reject = !((q == 0.0) || (u < p / q));
    }
    const unsigned int rej = __ballot_sync(0xffffffffu, reject);
    const int k = rej ? (__ffs(rej) - 1) : gb;
    if (i <= G && i != k) P.out_tokens[(size_t)b * (G + 1) + i] = i < k ? x : -1;
    if (i < G) {
      const bool evaluated = i < gb && i <= k;
      if (P.p_tok) P.p_tok[(size_t)b * G + i] = evaluated ? p : NAN;
      if (P.q_tok) P.q_tok[(size_t)b * G + i] = evaluated ? q : NAN;
    }
    const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
    if (i == 0) {
      P.num_accepted[b] = k;
      Decision d;
      d.k = k;
      d.reject = k < gb ? 1 : 0;
      d.mt = s_m[k];
      d.md = d.reject ? s_m[gb + 1 + k] : 0.0f;
      d.inv_st = (float)(1.0 / s_s[k]);
      d.rho = d.reject ? (float)(s_s[k] / s_s[gb + 1 + k]) : 0.0f;
      d.c_hi = tc.hi;
      d.c_lo = tc.lo;
      P.dec[b] = d;
      if (any) atomicOr(P.status, any);
      P.cnt_a[b] = 0;
      __threadfence();
      atomicExch(&P.ready[b], 1u);
    }
  }
  __syncthreads();
}

// Greedy decision: argmax per target row from the per-warp partials, then the
// first mismatch by warp ballot.
__device__ __noinline__ void decide_greedy(const Params& P, int b) {
  __shared__ int s_g[SV_MAX_GAMMA + 1];
  const int G = P.G, V = P.V, NC = P.NC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gb = clamp_gamma(P.gamma[b], G);
  unsigned int flags = (P.gamma[b] != gb) ? SV_STATUS_BAD_GAMMA : 0u;
  const int nparts = NC * kWarps;
  for (int r = warp; r <= gb; r += kWarps) {
    const float2* pr = P.stats + ((size_t)b * (2 * G + 1) + r) * P.stride_nc * kWarps;
    float v = -INFINITY;
    int idx = 0x7fffffff;
    for (int j = lane; j < nparts; j += 32) {
      const float2 mi = __ldcg(&pr[j]);
      argmax_combine(v, idx, mi.x, __float_as_int(mi.y));
    }
    warp_argmax(v, idx);
    if (lane == 0) {
      if (!isfinite(v)) flags |= SV_STATUS_NONFINITE_ROW;
      s_g[r] = (idx >= 0 && idx < V) ? idx : 0;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int i = lane;
    int x = 0;
    bool mismatch = false;
    if (i < gb) {
      x = P.tokens[(size_t)b * G + i];
      if (x < 0 || x >= V) flags |= SV_STATUS_BAD_TOKEN;
      mismatch = x != s_g[i];
    }
    const unsigned int mm = __ballot_sync(0xffffffffu, mismatch);
    const int k = mm ? (__ffs(mm) - 1) : gb;
    if (i <= G) P.out_tokens[(size_t)b * (G + 1) + i] = i < k ? x : (i == k ? s_g[k] : -1);
    const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
    if (i == 0) {
      P.num_accepted[b] = k;
      if (any) atomicOr(P.status, any);
      P.cnt_a[b] = 0;
    }
  }
  __syncthreads();
}

// Final draw for request b, run by the whole CTA that completed its last R item.
template <int EB>
__device__ __noinline__ void final_draw(const Params& P, int b) {
  __shared__ unsigned long long sh_scan[2 * kWarps + 1];
  __shared__ int sh_chunk, sh_usep, sh_tok;
  __shared__ unsigned long long sh_base, sh_target;
  constexpr int RE = kHalfBytes / EB;          // elements per R chunk
  constexpr int EPT = RE / kThreads;           // elements per thread in the scan
  const int G = P.G, V = P.V, NCR = P.NCR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Decision d = load_decision(&P.dec[b]);
  unsigned int flags = 0;
  const float u_s = sanitize_uniform(P.uniforms[(size_t)b * (G + 1) + G], flags);
  const ulonglong2* rp = P.resid + (size_t)b * P.stride_ncr;

  if (warp == 0) {
    unsigned long long tr = 0, tp = 0;
    for (int c = lane; c < NCR; c += 32) {
      const ulonglong2 w = __ldcg(&rp[c]);
      tr += w.x;
      tp += w.y;
    }
    tr = warp_sum_u64(tr);
    tp = warp_sum_u64(tp);
    const int usep = (tr == 0ull);  // residual vanished: draw from p_k
    const unsigned long long S = usep ? tp : tr;
    const unsigned long long target = scaled_target(u_s, S);
    unsigned long long carry = 0, base = 0;
    int found = -1;
    for (int c0 = 0; c0 < NCR && found < 0; c0 += 32) {
      const int c = c0 + lane;
      unsigned long long w = 0;
      if (c < NCR) {
        const ulonglong2 ww = __ldcg(&rp[c]);
        w = usep ? ww.y : ww.x;
      }
      unsigned long long incl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned int hit = __ballot_sync(0xffffffffu, c < NCR && carry + incl > target);
      if (hit) {
        const int l = __ffs(hit) - 1;
        found = c0 + l;
        base = carry + __shfl_sync(0xffffffffu, incl - w, l);
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      sh_chunk = found;
      sh_usep = usep;
      sh_base = base;
      sh_target = target;
      sh_tok = -1;
    }
  }
  __syncthreads();
  const int cs = sh_chunk;
  if (cs >= 0) {
    ResidC kc;
    kc.mt = d.mt; kc.md = d.md; kc.inv_st = d.inv_st; kc.rho = d.rho;
    kc.hi = d.c_hi; kc.lo = d.c_lo; kc.reject = d.reject;
    const char* trow = P.target + target_row(b, d.k, G, V) * EB;
    const char* drow = d.reject ? P.draft + draft_row(b, d.k, G, V) * EB : nullptr;
    const int e0 = (int)threadIdx.x * EPT;
    const int usep = sh_usep;
    // weight of element j of this thread's run (recomputed, bit-identical)
    auto weight = [&](int j) -> unsigned long long {
      const size_t e = (size_t)cs * RE + (size_t)(e0 + j);
      unsigned long long wr = 0, wp = 0;
      if (e < (size_t)V) {
        const float zt = load_elem<EB>(trow, e);
        const float zd = drow ? load_elem<EB>(drow, e) : -INFINITY;
        resid_weights(zt, zd, kc, wr, wp);
      }
      return usep ? wp : wr;
    };
    unsigned long long tsum = 0;
#pragma unroll 4
    for (int j = 0; j < EPT; ++j) tsum += weight(j);
    unsigned long long total;
    const unsigned long long excl = block_exclusive_scan(tsum, sh_scan, &total);
    const unsigned long long target = sh_target;
    unsigned long long run = sh_base + excl;
    if (run <= target && run + tsum > target) {
      for (int j = 0; j < EPT; ++j) {
        const unsigned long long nxt = run + weight(j);
        if (run <= target && nxt > target) {
          sh_tok = cs * RE + e0 + j;
          break;
        }
        run = nxt;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tok = sh_tok;
    if (tok < 0) {
      flags |= SV_STATUS_INTERNAL;
      tok = V - 1;
    }
    P.out_tokens[(size_t)b * (G + 1) + d.k] = tok;
    if (flags) atomicOr(P.status, flags);
    P.cnt_r[b] = 0;
    P.ready[b] = 0;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Work-item order and decoding (thread 0)
// ---------------------------------------------------------------------------
struct Sched {
  const int* rowpre;  // [B+1] exclusive prefix of rows per request (shared memory)
  int B, L, NC, NCR;
  int mode;
  unsigned int total;
};

// start of segment k: A items of requests < k plus R items of requests < k - L
__device__ __forceinline__ unsigned int seg_start(const Sched& s, int k) {
  const int r = k - s.L;
  return (unsigned int)s.rowpre[k] * s.NC + (r > 0 ? (unsigned int)r * s.NCR : 0u);
}

// Fill `out` for item j.  For R items whose request has not been decided
// yet, returns KIND_RWAIT (nothing is read from the decision).
template <int EB>
__device__ __noinline__ void decode_item(const Params& P, const Sched& s, unsigned int j, Slot& out,
                            int& kcache) {
  if (j >= s.total) {
    out.kind = KIND_EXIT;
    return;
  }
  int req = -1, c = 0;
  bool is_r = false;
  if (s.mode == MODE_SAMPLE && j >= seg_start(s, s.B)) {
    const unsigned int t = j - seg_start(s, s.B);
    req = (s.B > s.L ? s.B - s.L : 0) + (int)(t / s.NCR);
    c = (int)(t % s.NCR);
    is_r = true;
  } else {
    // largest k with seg_start(k) <= j, searching up from the last answer
    int lo = kcache, hi = s.B - 1;
    if (seg_start(s, lo) > j) lo = 0;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (seg_start(s, mid) <= j) lo = mid; else hi = mid - 1;
    }
    kcache = lo;
    const unsigned int off = j - seg_start(s, lo);
    const unsigned int na = (unsigned int)(s.rowpre[lo + 1] - s.rowpre[lo]) * s.NC;
    if (off < na) {
      const int G = P.G, V = P.V;
      const int row = (int)(off / s.NC);
      c = (int)(off % s.NC);
      const int gb = (s.mode == MODE_SAMPLE) ? (s.rowpre[lo + 1] - s.rowpre[lo] - 1) / 2
                                             : (s.rowpre[lo + 1] - s.rowpre[lo] - 1);
      size_t roff;
      if (row <= gb) {
        out.pslot = row;
        roff = target_row(lo, row, G, V);
      } else {
        const int i = row - gb - 1;
        out.pslot = G + 1 + i;
        roff = draft_row(lo, i, G, V);
      }
      constexpr int AE = kTileBytes / EB;
      const char* base = row <= gb ? P.target : P.draft;
      out.kind = KIND_A;
      out.b = lo;
      out.c = c;
      out.n = min(AE, V - c * AE);
      out.p0 = base + (roff + (size_t)c * AE) * EB;
      out.p1 = nullptr;
      out.aligned = (reinterpret_cast<uintptr_t>(out.p0) & 15) == 0;
      if (s.mode == MODE_SAMPLE) {
        unsigned int fl = 0;
        const TempC tc = temp_consts(sanitize_temperature(P.temperature[lo], fl));
        out.c_hi = tc.hi;
        out.c_lo = tc.lo;
      }
      return;
    }
    req = lo - s.L;
    c = (int)(off - na);
    is_r = true;
  }
  (void)is_r;
  out.b = req;
  out.c = c;
  if (!ld_acquire(&P.ready[req])) {
    out.kind = KIND_RWAIT;
    return;
  }
  // decision published: read it and build the R item
  const Decision d = load_decision(&P.dec[req]);
  const int G = P.G, V = P.V;
  const int k = d.k < 0 ? 0 : (d.k > G ? G : d.k);
  const int reject = (d.reject && k < G) ? 1 : 0;
  constexpr int RE = kHalfBytes / EB;
  out.kind = KIND_R;
  out.pslot = k;
  out.reject = reject;
  out.n = min(RE, V - c * RE);
  out.p0 = P.target + (target_row(req, k, G, V) + (size_t)c * RE) * EB;
  out.p1 = reject ? P.draft + (draft_row(req, k, G, V) + (size_t)c * RE) * EB : nullptr;
  out.aligned = ((reinterpret_cast<uintptr_t>(out.p0) | reinterpret_cast<uintptr_t>(out.p1)) & 15) == 0;
  out.mt = d.mt;
  out.md = d.md;
  out.inv_st = d.inv_st;
  out.rho = d.rho;
  out.c_hi = d.c_hi;
  out.c_lo = d.c_lo;
}

// ---------------------------------------------------------------------------
// Item compute
// ---------------------------------------------------------------------------
template <int EB>
__device__ __forceinline__ void issue_loads(const Slot& s, uint4 (&buf)[kVecA]) {
  if (s.kind == KIND_A) {
    load_tile<EB, kVecA>(buf, s.p0, s.n, s.aligned);
  } else if (s.kind == KIND_R) {
    load_tile<EB, kVecA / 2>(buf, s.p0, s.n, s.aligned);
    if (s.p1) load_tile<EB, kVecA / 2>(buf + kVecA / 2, s.p1, s.n, s.aligned);
    else fill_neg_inf(buf + kVecA / 2, kVecA / 2, EB);
  }
}

template <int EB, int MODE>
__device__ __forceinline__ void compute_a(const Params& P, const Slot& s,
                                          const uint4 (&buf)[kVecA]) {
  constexpr int VEC = 16 / EB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float2* part = P.stats + (((size_t)s.b * (2 * P.G + 1) + s.pslot) * P.stride_nc + s.c) * kWarps + warp;
  if (MODE == MODE_SAMPLE) {
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kVecA; ++k)
#pragma unroll
      for (int j = 0; j < VEC; ++j) m = fmaxf(m, vec_elem<EB>(buf[k], j));
    m = warp_max(m);
    float sum = 0.0f;
    if (m > -INFINITY) {
#pragma unroll
      for (int k = 0; k < kVecA; ++k) {
        float e[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) e[j] = ex2_approx(exp_arg(vec_elem<EB>(buf[k], j), m, s.c_hi, s.c_lo));
#pragma unroll
        for (int w = VEC; w > 1; w >>= 1)
#pragma unroll
          for (int j = 0; j < w / 2; ++j) e[j] = e[2 * j] + e[2 * j + 1];
        sum += e[0];
      }
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      *part = make_float2(m, sum);
      __threadfence();
    }
  } else {
    constexpr int AE = kTileBytes / EB;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int k = 0; k < kVecA; ++k)
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        const int e = ((int)threadIdx.x + k * kThreads) * VEC + j;
        argmax_combine(bv, bi, vec_elem<EB>(buf[k], j), s.c * AE + e);
      }
    warp_argmax(bv, bi);
    if (lane == 0) {
      *part = make_float2(bv, __int_as_float(bi));
      __threadfence();
    }
  }
}

template <int EB>
__device__ __forceinline__ void compute_r(const Slot& s, const uint4 (&buf)[kVecA],
                                          unsigned long long* sh_r, unsigned long long* sh_p) {
  constexpr int VEC = 16 / EB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ResidC kc;
  kc.mt = s.mt; kc.md = s.md; kc.inv_st = s.inv_st; kc.rho = s.rho;
  kc.hi = s.c_hi; kc.lo = s.c_lo; kc.reject = s.reject;
  unsigned long long sr = 0, sp = 0;
#pragma unroll
  for (int k = 0; k < kVecA / 2; ++k)
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      unsigned long long wr, wp;
      resid_weights(vec_elem<EB>(buf[k], j), vec_elem<EB>(buf[kVecA / 2 + k], j), kc, wr, wp);
      sr += wr;
      sp += wp;
    }
  sr = warp_sum_u64(sr);
  sp = warp_sum_u64(sp);
  if (lane == 0) {
    sh_r[warp] = sr;
    sh_p[warp] = sp;
  }
}

// ---------------------------------------------------------------------------
// The persistent kernel
// ---------------------------------------------------------------------------
struct Pending {  // thread 0's record of the last item's arrival
  int kind;       // KIND_A / KIND_R / -1 (none)
  int b;
  unsigned int old, total;
};

template <int EB, int MODE>
__device__ __forceinline__ void run_pending(const Params& P, const int* work) {
  // work[0] = kind of completed request (-1 none), work[1] = request
  if (work[0] == KIND_A) {
    if (MODE == MODE_SAMPLE) decide_sample<EB>(P, work[1]);
    else decide_greedy(P, work[1]);
  } else if (work[0] == KIND_R) {
    final_draw<EB>(P, work[1]);
  }
}

template <int EB, int MODE>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(Params P) {
  extern __shared__ int rowpre[];  // [B + 1]
  __shared__ Slot slots[3];
  __shared__ int sh_work[2][2];
  __shared__ unsigned long long sh_r[2][kWarps], sh_p[2][kWarps];
  __shared__ int sh_carry;
  const int tid = threadIdx.x;
  const int G = P.G, B = P.B;

  // rows per request -> exclusive prefix in shared memory
  if (tid == 0) {
    rowpre[0] = 0;
    sh_carry = 0;
  }
  __syncthreads();
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + tid;
    int v = 0;
    if (b < B) {
      const int gb = clamp_gamma(P.gamma[b], G);
      v = MODE == MODE_SAMPLE ? 2 * gb + 1 : gb + 1;
    }
    const int lane = tid & 31, warp = tid >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __shared__ int wsum[kWarps];
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int off = sh_carry;
    for (int w = 0; w < warp; ++w) off += wsum[w];
    if (b < B) rowpre[b + 1] = off + incl;
    __syncthreads();
    if (tid == kThreads - 1) sh_carry = off + incl;
    __syncthreads();
  }

  Sched sc;
  sc.rowpre = rowpre;
  sc.B = B;
  sc.NC = P.NC;
  sc.NCR = MODE == MODE_SAMPLE ? P.NCR : 0;
  sc.mode = MODE;
  {
    const unsigned int totalA = (unsigned int)rowpre[B] * P.NC;
    int L = 1;
    if (MODE == MODE_SAMPLE) {
      // keep R items about three grids of items behind their decisions
      const double per_req = (double)totalA / (double)B;
      L = (int)ceil(3.0 * gridDim.x / per_req);
      if (L < 1) L = 1;
    }
    sc.L = L;
    sc.total = totalA + (MODE == MODE_SAMPLE ? (unsigned int)B * P.NCR : 0u);
  }

  uint4 bufX[kVecA], bufY[kVecA];
  Pending pend;
  pend.kind = -1;
  int kcache = 0;
  unsigned int flags0 = 0;
  if (tid == 0) {
    decode_item<EB>(P, sc, atomicAdd(P.next_item, 1u), slots[0], kcache);
    decode_item<EB>(P, sc, atomicAdd(P.next_item, 1u), slots[1], kcache);
    sh_work[0][0] = sh_work[1][0] = -1;
  }
  __syncthreads();
  issue_loads<EB>(slots[0], bufX);

  int cur = 0, parity = 0;
  // One iteration: claim item n+2, prefetch item n+1, compute item n, then
  // publish item n's arrival (its follow-up work runs one iteration later).
  auto step = [&](uint4 (&X)[kVecA], uint4 (&Y)[kVecA]) -> bool {
    Slot& s = slots[cur];
    if (s.kind == KIND_EXIT) return false;
    if (s.kind == KIND_RWAIT) {
      // Finish everything held (the previous item's follow-up) before waiting.
      if (tid == 0) {
        int wk = -1;
        if (pend.kind == KIND_A && pend.old == pend.total - 1) wk = KIND_A;
        if (pend.kind == KIND_R && pend.old == pend.total - 1) wk = KIND_R;
        if (wk >= 0) __threadfence();
        sh_work[parity][0] = wk;
        sh_work[parity][1] = pend.b;
        pend.kind = -1;
      }
      __syncthreads();
      run_pending<EB, MODE>(P, sh_work[parity]);
      if (tid == 0) {
        unsigned int it = 0;
        while (!ld_acquire(&P.ready[s.b])) {
          if (++it > kSpinLimit) {
            flags0 |= SV_STATUS_TIMEOUT;
            break;
          }
          __nanosleep(256);
        }
      }
      // rebuild the item from the now-published decision
      if (tid == 0) {
        if (!(flags0 & SV_STATUS_TIMEOUT)) {
          const Decision d = load_decision(&P.dec[s.b]);
          const int V = P.V;
          const int k = d.k < 0 ? 0 : (d.k > G ? G : d.k);
          const int reject = (d.reject && k < G) ? 1 : 0;
          constexpr int RE = kHalfBytes / EB;
          s.kind = KIND_R;
          s.pslot = k;
          s.reject = reject;
          s.n = min(RE, V - s.c * RE);
          s.p0 = P.target + (target_row(s.b, k, G, V) + (size_t)s.c * RE) * EB;
          s.p1 = reject ? P.draft + (draft_row(s.b, k, G, V) + (size_t)s.c * RE) * EB : nullptr;
          s.aligned = ((reinterpret_cast<uintptr_t>(s.p0) | reinterpret_cast<uintptr_t>(s.p1)) & 15) == 0;
          s.mt = d.mt; s.md = d.md; s.inv_st = d.inv_st; s.rho = d.rho;
          s.c_hi = d.c_hi; s.c_lo = d.c_lo;
        } else {
          s.kind = KIND_EXIT;  // give up: the status word reports it
        }
      }
      __syncthreads();
      if (s.kind == KIND_EXIT) return false;
      issue_loads<EB>(s, X);
    }

    unsigned int ticket = 0;
    if (tid == 0) ticket = atomicAdd(P.next_item, 1u);
    Slot& sn = slots[(cur + 1) % 3];
    issue_loads<EB>(sn, Y);

    if (s.kind == KIND_A) compute_a<EB, MODE>(P, s, X);
    else compute_r<EB>(s, X, sh_r[parity], sh_p[parity]);

    if (tid == 0) {
      decode_item<EB>(P, sc, ticket, slots[(cur + 2) % 3], kcache);
      int wk = -1;
      if (pend.kind >= 0 && pend.old == pend.total - 1) {
        wk = pend.kind;
        __threadfence();
      }
      sh_work[parity][0] = wk;
      sh_work[parity][1] = pend.b;
      pend.kind = -1;
    }
    __syncthreads();
    run_pending<EB, MODE>(P, sh_work[parity]);
    if (tid == 0) {
      if (s.kind == KIND_A) {
        const int rows = rowpre[s.b + 1] - rowpre[s.b];
        pend.kind = KIND_A;
        pend.b = s.b;
        pend.total = (unsigned int)rows * P.NC;
        pend.old = atomicAdd(&P.cnt_a[s.b], 1u);
      } else {
        unsigned long long tr = 0, tp = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          tr += sh_r[parity][w];
          tp += sh_p[parity][w];
        }
        P.resid[(size_t)s.b * P.stride_ncr + s.c] = make_ulonglong2(tr, tp);
        __threadfence();
        pend.kind = KIND_R;
        pend.b = s.b;
        pend.total = (unsigned int)P.NCR;
        pend.old = atomicAdd(&P.cnt_r[s.b], 1u);
      }
    }
    cur = (cur + 1) % 3;
    parity ^= 1;
    return true;
  };

  for (;;) {
    if (!step(bufX, bufY)) break;
    if (!step(bufY, bufX)) break;
  }

  // drain the last item's follow-up, then leave; the last CTA out resets the
  // shared counters so the workspace is zeroed for the next call
  if (tid == 0) {
    int wk = -1;
    if (pend.kind >= 0 && pend.old == pend.total - 1) {
      wk = pend.kind;
      __threadfence();
    }
    sh_work[parity][0] = wk;
    sh_work[parity][1] = pend.b;
  }
  __syncthreads();
  run_pending<EB, MODE>(P, sh_work[parity]);
  if (tid == 0) {
    if (flags0) atomicOr(P.status, flags0);
    __threadfence();
    const unsigned int done = atomicAdd(P.exit_count, 1u);
    if (done == gridDim.x - 1) {
      *P.next_item = 0;
      *P.exit_count = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int check_scalars(sv_dtype dtype, int B, int G, int V) {
  if (B < 0 || G < 0 || G > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB) return SV_ERR_SCALAR;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_SCALAR;
  return SV_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int EB, int MODE>
int grid_size(size_t smem) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<EB, MODE>, kThreads,
                                                    smem) != cudaSuccess)
    return 0;
  return sms * (per_sm > 0 ? per_sm : 1);
}

template <int EB, int MODE>
int launch(Params P, const Layout& L, char* ws, cudaStream_t stream) {
  // requests are processed in launches of at most kMaxBatch
  const int B = P.B;
  for (int b0 = 0; b0 < B; b0 += kMaxBatch) {
    Params Q = P;
    Q.B = B - b0 < kMaxBatch ? B - b0 : kMaxBatch;
    const size_t G = (size_t)P.G, V = (size_t)P.V;
    Q.target = P.target + (size_t)b0 * (G + 1) * V * EB;
    Q.draft = P.draft ? P.draft + (size_t)b0 * G * V * EB : nullptr;
    Q.tokens = P.tokens ? P.tokens + (size_t)b0 * G : nullptr;
    Q.gamma = P.gamma + b0;
    Q.uniforms = P.uniforms ? P.uniforms + (size_t)b0 * (G + 1) : nullptr;
    Q.temperature = P.temperature ? P.temperature + b0 : nullptr;
    Q.out_tokens = P.out_tokens + (size_t)b0 * (G + 1);
    Q.num_accepted = P.num_accepted + b0;
    Q.p_tok = P.p_tok ? P.p_tok + (size_t)b0 * G : nullptr;
    Q.q_tok = P.q_tok ? P.q_tok + (size_t)b0 * G : nullptr;
    Q.cnt_a = P.cnt_a + b0;
    Q.cnt_r = P.cnt_r + b0;
    Q.ready = P.ready + b0;
    Q.dec = P.dec + b0;
    Q.stats = P.stats + (size_t)b0 * (2 * G + 1) * P.stride_nc * kWarps;
    Q.resid = P.resid + (size_t)b0 * P.stride_ncr;
    const size_t smem = (size_t)(Q.B + 1) * sizeof(int);
    const int grid = grid_size<EB, MODE>(smem);
    if (grid <= 0) return SV_ERR_CUDA;
    verify_kernel<EB, MODE><<<grid, kThreads, smem, stream>>>(Q);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  (void)L;
  (void)ws;
  return SV_OK;
}

int fill_params(Params& P, const void* target, const void* draft, sv_dtype dtype, int B, int G,
                int V, const int32_t* tokens, const int32_t* gamma, const float* uniforms,
                const float* temperature, int32_t* out_tokens, int32_t* num_accepted,
                double* p_tok, double* q_tok, void* ws, size_t ws_bytes, Layout& L) {
  L = make_layout(B, G, V);
  if (ws_bytes < L.total) return SV_ERR_WORKSPACE;
  const size_t eb = dtype == SV_BF16 ? 2 : 4;
  if (!aligned(target, eb) || (draft && !aligned(draft, eb))) return SV_ERR_ALIGN;
  if (!aligned(tokens, 4) || !aligned(gamma, 4) || !aligned(uniforms, 4) ||
      !aligned(temperature, 4) || !aligned(out_tokens, 4) || !aligned(num_accepted, 4))
    return SV_ERR_ALIGN;
  if (!aligned(p_tok, 8) || !aligned(q_tok, 8) || !aligned(ws, 256)) return SV_ERR_ALIGN;
  char* w = static_cast<char*>(ws);
  P.target = static_cast<const char*>(target);
  P.draft = static_cast<const char*>(draft);
  P.B = B;
  P.G = G;
  P.V = V;
  P.NC = (int)((V + kTileBytes / eb - 1) / (kTileBytes / eb));
  P.NCR = (int)((V + kHalfBytes / eb - 1) / (kHalfBytes / eb));
  P.stride_nc = L.NC;
  P.stride_ncr = L.NCR;
  P.tokens = tokens;
  P.gamma = gamma;
  P.uniforms = uniforms;
  P.temperature = temperature;
  P.out_tokens = out_tokens;
  P.num_accepted = num_accepted;
  P.p_tok = p_tok;
  P.q_tok = q_tok;
  P.status = reinterpret_cast<unsigned int*>(w + L.status);
  P.next_item = reinterpret_cast<unsigned int*>(w + L.next_item);
  P.exit_count = reinterpret_cast<unsigned int*>(w + L.exit_count);
  P.cnt_a = reinterpret_cast<unsigned int*>(w + L.cnt_a);
  P.cnt_r = reinterpret_cast<unsigned int*>(w + L.cnt_r);
  P.ready = reinterpret_cast<unsigned int*>(w + L.ready);
  P.dec = reinterpret_cast<Decision*>(w + L.dec);
  P.stats = reinterpret_cast<float2*>(w + L.stats);
  P.resid = reinterpret_cast<ulonglong2*>(w + L.resid);
  return SV_OK;
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int B, int G, int V) {
  if (check_scalars(SV_BF16, B, G, V) != SV_OK) return 0;
  return make_layout(B, G, V).total;
}

int spec_verify_sample(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                       int B, int G, int V, const int32_t* draft_tokens,
                       const int32_t* gamma, const float* uniforms, const float* temperature,
                       int32_t* out_tokens, int32_t* num_accepted, double* p_tok,
                       double* q_tok, void* workspace, size_t ws_bytes, sv_stream_t stream) {
  int rc = check_scalars(dtype, B, G, V);
  if (rc) return rc;
  if (!target_logits || !gamma || !uniforms || !temperature || !out_tokens || !num_accepted ||
      !workspace)
    return SV_ERR_NULL;
  if (G > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_NULL;
  Params P;
  Layout L;
  rc = fill_params(P, target_logits, draft_logits, dtype, B, G, V, draft_tokens, gamma, uniforms,
                   temperature, out_tokens, num_accepted, p_tok, q_tok, workspace, ws_bytes, L);
  if (rc) return rc;
  if (B == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  return dtype == SV_BF16 ? launch<2, MODE_SAMPLE>(P, L, ws, s)
                          : launch<4, MODE_SAMPLE>(P, L, ws, s);
}

int spec_verify_greedy(const void* target_logits, sv_dtype dtype, int B, int G, int V,
                       const int32_t* draft_tokens, const int32_t* gamma, int32_t* out_tokens,
                       int32_t* num_accepted, void* workspace, size_t ws_bytes,
                       sv_stream_t stream) {
  int rc = check_scalars(dtype, B, G, V);
  if (rc) return rc;
  if (!target_logits || !gamma || !out_tokens || !num_accepted || !workspace)
    return SV_ERR_NULL;
  if (G > 0 && !draft_tokens) return SV_ERR_NULL;
  Params P;
  Layout L;
  rc = fill_params(P, target_logits, nullptr, dtype, B, G, V, draft_tokens, gamma, nullptr,
                   nullptr, out_tokens, num_accepted, nullptr, nullptr, workspace, ws_bytes, L);
  if (rc) return rc;
  if (B == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  return dtype == SV_BF16 ? launch<2, MODE_GREEDY>(P, L, ws, s)
                          : launch<4, MODE_GREEDY>(P, L, ws, s);
}

int spec_verify_status(void* workspace, sv_stream_t stream, uint32_t* status_host) {
  if (!workspace || !status_host) return SV_ERR_NULL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The status word sits at offset 0 of every workspace layout.
  if (cudaMemcpyAsync(status_host, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return SV_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

const char* spec_verify_strerror(int code) {
  switch (code) {
    case SV_OK: return "success";
    case SV_ERR_SCALAR: return "invalid size or dtype argument";
    case SV_ERR_NULL: return "a required pointer is NULL";
    case SV_ERR_ALIGN: return "a pointer is not suitably aligned";
    case SV_ERR_WORKSPACE: return "workspace smaller than spec_verify_workspace_size()";
    case SV_ERR_CUDA: return "CUDA launch or copy failed";
    default: return "unknown error code";
  }
}

}  // extern "C"
