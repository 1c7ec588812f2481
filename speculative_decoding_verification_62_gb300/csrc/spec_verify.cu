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
// One persistent kernel per call, one CTA of 12 warps per SM.  Work items, in
// one fixed order:
//   A items  8 KB of one logit row: max and sum of exp2((z - max) log2(e)/T)
//            (sampling) or argmax (greedy) -> one partial per item.  All A
//            items come first, request-major.
//   R items  4 KB of target row k and the same 4 KB of draft row k of one
//            request (sampling): fixed-point (2^-39) sums of the residual
//            max(0, p_k - q_k) and of p_k -> one partial per item.  They form
//            a tail that starts a few requests before the end and walks
//            backwards, so the first ones re-read rows still in L2.
// Every warp runs its own pipeline: it claims small batches of items from one
// global counter (the next batch is claimed while the current one runs, and
// its lanes decode a batch in parallel), keeps kNB TMA bulk copies
// (cp.async.bulk) in flight into private shared-memory buffers, each tracked
// by one mbarrier, and processes the items in order.  Arrivals are counted
// per request with one acquire-release atomic per batch; the warp that
// completes a request's A items runs its decision (float-float normalisers,
// float64 acceptance ratios, warp-ballot first reject) and publishes it; the
// warp that completes its R items locates the chunk holding u*S and scans
// only that chunk for the token.  An R item whose request is not decided yet
// is deferred while other items remain; a warp waits for a decision only
// with its pipeline drained and its arrivals published, and only in the R
// tail (it has then issued all its A items), so every wait ends.  Each wait
// is also bounded (2 s) and sets SV_STATUS_TIMEOUT.  Counters are reset by
// their last user, so the workspace stays zeroed.
//
// Numerics: inputs widen exactly to float32.  Exponent arguments use a
// two-term log2(e)/T (hi + lo); exp2 is the SFU's ex2.approx; sums inside an
// item are float32, sums across items float64.  The acceptance ratio is
// formed in float64.  The residual CDF is summed in exact 64-bit fixed point,
// so chunk sums and the final in-chunk scan agree bit for bit.

#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>
#include <math.h>
#include <float.h>

#include "spec_verify.h"

namespace {

#ifndef SV_WARPS
#define SV_WARPS 12
#endif
#ifndef SV_BUFFERS
#define SV_BUFFERS 2
#endif
constexpr int kWarps = SV_WARPS;                      // warps per CTA (one CTA per SM)
constexpr int kThreads = 32 * kWarps;
constexpr int kNB = SV_BUFFERS;                       // TMA buffers per warp
constexpr int kItemBytes = 8192;                      // A item: 8 KB of one row
constexpr int kHalfBytes = kItemBytes / 2;            // R item: 2 KB of each of two rows
constexpr int kMaxBatch = 4096;                       // requests per launch (smem prefix)
constexpr int kMaxK = 8;                              // work items per claimed batch
constexpr unsigned int kBatchDiv = 4;                 // batches per warp's share, at least
constexpr int kDefer = 32;                            // deferred R items per warp
constexpr unsigned long long kWaitNs = 2000000000ull; // every wait gives up after 2 s
constexpr float kFix = 549755813888.0f;               // 2^39: fixed-point scale of probabilities
constexpr float kLog2eHi = 1.44269502162933349609375f;      // float nearest log2(e)
constexpr float kLog2eLo = 1.925963033500011e-08f;          // log2(e) - kLog2eHi

enum { KIND_A = 0, KIND_R = 1 };
enum { MODE_SAMPLE = 0, MODE_GREEDY = 1 };

// ---------------------------------------------------------------------------
// Workspace
// ---------------------------------------------------------------------------
struct Decision {      // per request, published by the deciding warp
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
  L.NC = (V + kItemBytes / 4 - 1) / (kItemBytes / 4);
  L.NCR = (V + kHalfBytes / 4 - 1) / (kHalfBytes / 4);
  L.status = 0;
  L.next_item = 64;
  L.exit_count = 128;
  size_t off = 256;
  L.cnt_a = off; off = align256(off + (size_t)B * 4);
  L.cnt_r = off; off = align256(off + (size_t)B * 4);
  L.ready = off; off = align256(off + (size_t)B * 4);
  L.dec = off;   off = align256(off + (size_t)B * sizeof(Decision));
  L.stats = off; off = align256(off + (size_t)B * (2 * G + 1) * L.NC * sizeof(float2));
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
  unsigned int* next_item;   // next work item to claim
  unsigned int* exit_count;
  unsigned int* cnt_a;       // [B] A items completed
  unsigned int* cnt_r;       // [B] R items completed
  unsigned int* ready;       // [B] 1 once the request's decision is published
  Decision* dec;
  float2* stats;       // [B][2G+1][stride_nc]: (max, sum) or (max, argmax bits)
  ulonglong2* resid;   // [B][stride_ncr]: (residual sum, p sum)
};

// A decoded work item (one per lane of a claimed batch; stored per buffer).
struct Meta {
  int kind;
  int b;
  int pslot;    // A: partial row slot
  int c;        // chunk index
  int n;        // valid elements (A: in the item; R: per row)
  int direct;   // 1: bytes not copied (unaligned); read them from global memory
  int reject;   // R
  int pad;
  const char* p0;  // A: item start; R: target half
  const char* p1;  // R: draft half, or null for the bonus draw
  float mt, md, inv_st, rho, c_hi, c_lo;
};

// ---------------------------------------------------------------------------
// PTX helpers: mbarriers, bulk copies, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > kWaitNs) return false;
  }
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
  return v;
}
// Atomic add with acquire-release semantics: publishes this thread's earlier
// writes and, for the last arriver, makes the other arrivers' writes visible.
__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_release(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed arithmetic: max of two bf16 pairs (exact), and pairs of float32
// lanes in one 64-bit register (each lane an ordinary IEEE round-to-nearest
// operation).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// the two bf16 logits of a 32-bit word as a float32 pair (low element first)
__device__ __forceinline__ unsigned long long bf16x2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ float bf16x2_hmax(uint32_t w) {
  return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// per-half equality of two bf16 pairs (0xffff in each equal half)
__device__ __forceinline__ uint32_t bf16x2_eq(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t vec_word(const uint4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
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

// element j of a 16-byte vector holding 16/EB logits
template <int EB>
__device__ __forceinline__ float vec_elem(const uint4& v, int j) {
  const uint32_t w = j < (EB == 2 ? 2 : 1) ? v.x : j < (EB == 2 ? 4 : 2) ? v.y
                   : j < (EB == 2 ? 6 : 3) ? v.z : v.w;
  if (EB == 2) return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  return __uint_as_float(w);
}

// a 16-byte vector of -inf logits
__device__ __forceinline__ uint4 neg_inf_vec(int eb) {
  const uint32_t f = eb == 2 ? 0xff80ff80u : 0xff800000u;
  return make_uint4(f, f, f, f);
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
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
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

// Float-float (hi + lo) sums: about 48 bits of precision from float32 adds.
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return FF{s, e};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const FF s = ff_two_sum(a.hi, b.hi);
  const float e = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  return ff_two_sum(s.hi, e);
}
__device__ __forceinline__ FF warp_sum_ff(FF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF w;
    w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
    w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
    v = ff_add(v, w);
  }
  return v;
}

// ---------------------------------------------------------------------------
// Per-request decision (sampling), run by one warp: the one that completed
// the request's last A item.
// ---------------------------------------------------------------------------
template <int EB>
__device__ __noinline__ void decide_sample(const Params& P, int b) {
  const int G = P.G, V = P.V, NC = P.NC;
  const int lane = threadIdx.x & 31;
  const int gb = clamp_gamma(P.gamma[b], G);
  unsigned int flags = (P.gamma[b] != gb) ? SV_STATUS_BAD_GAMMA : 0u;
  const float T = sanitize_temperature(P.temperature[b], flags);
  const TempC tc = temp_consts(T);
  const double cd = (double)tc.hi + (double)tc.lo;
  const int nrows = 2 * gb + 1;

  // Row maximum M and normaliser S = sum_c s_c 2^((m_c - M) c) over the
  // per-item partials, summed in float-float.  Lane (r & 31) keeps row r in
  // slot r >> 5.  Four rows at a time, each lane loading chunks lane and
  // lane + 32, so the loads of a group are in flight together.
  float rowM[2] = {-INFINITY, -INFINITY};
  double rowS[2] = {0.0, 0.0};
  const float2 none = make_float2(-INFINITY, 0.0f);
  for (int r0 = 0; r0 < nrows; r0 += 4) {
    float2 v[4][2];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int r = r0 + g;
      const int slot = r <= gb ? r : (G + 1 + (r - gb - 1));
      const float2* pr = P.stats + ((size_t)b * (2 * G + 1) + slot) * P.stride_nc;
      v[g][0] = (r < nrows && lane < NC) ? __ldcg(&pr[lane]) : none;
      v[g][1] = (r < nrows && lane + 32 < NC) ? __ldcg(&pr[lane + 32]) : none;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int r = r0 + g;
      if (r >= nrows) break;
      const int slot = r <= gb ? r : (G + 1 + (r - gb - 1));
      const float2* pr = P.stats + ((size_t)b * (2 * G + 1) + slot) * P.stride_nc;
      float M = fmaxf(v[g][0].x, v[g][1].x);
      for (int c = lane + 64; c < NC; c += 32) M = fmaxf(M, __ldcg(&pr[c]).x);
      M = warp_max(M);
      FF S{0.0f, 0.0f};
      if (M > -INFINITY) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (v[g][h].x > -INFINITY)
            S = ff_add(S, FF{__fmul_rn(v[g][h].y, ex2_approx(exp_arg(v[g][h].x, M, tc.hi, tc.lo))), 0.0f});
        for (int c = lane + 64; c < NC; c += 32) {
          const float2 ms = __ldcg(&pr[c]);
          if (ms.x > -INFINITY)
            S = ff_add(S, FF{__fmul_rn(ms.y, ex2_approx(exp_arg(ms.x, M, tc.hi, tc.lo))), 0.0f});
        }
      }
      S = warp_sum_ff(S);
      const double Sd = (double)S.hi + (double)S.lo;
      if (!isfinite(M) || !(Sd > 0.0)) flags |= SV_STATUS_NONFINITE_ROW;
      if (lane == (r & 31)) {
        rowM[r >> 5] = M;
        rowS[r >> 5] = Sd;
      }
    }
  }
  // row r's statistics, fetched from lane r & 31
  auto row_m = [&](int r) {
    const float a = __shfl_sync(0xffffffffu, rowM[0], r & 31);
    const float c = __shfl_sync(0xffffffffu, rowM[1], r & 31);
    return r < 32 ? a : c;
  };
  auto row_s = [&](int r) {
    const double a = __shfl_sync(0xffffffffu, rowS[0], r & 31);
    const double c = __shfl_sync(0xffffffffu, rowS[1], r & 31);
    return r < 32 ? a : c;
  };

  // Acceptance test per position (lane i), then the first-reject ballot.
  const int i = lane;
  const int ri = i < gb ? i : 0;
  const float mt_i = row_m(ri), md_i = row_m(gb + 1 + ri);
  const double st_i = row_s(ri), sd_i = row_s(gb + 1 + ri);
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
    const double et = ((double)zt - (double)mt_i) * cd;  // log2 of S_t p(x)
    const double ed = ((double)zd - (double)md_i) * cd;  // log2 of S_d q(x)
    const double u = (double)sanitize_uniform(P.uniforms[(size_t)b * (G + 1) + i], flags);
    // ratio p/q = 2^(et - ed) * S_d / S_t.  A draft probability q(x) that is
    // 0 in float64 (a -inf logit, or one far enough below the maximum to
    // underflow) accepts.
    const bool qzero = ed == -INFINITY || (ed < -1000.0 && exp2(ed) / sd_i == 0.0);
    const double ratio = exp2(et - ed) * (sd_i / st_i);
    reject = !(qzero || (u < ratio));
    if (P.p_tok || P.q_tok) {
      p = exp2(et) / st_i;
      q = exp2(ed) / sd_i;
    }
  }
  const unsigned int rej = __ballot_sync(0xffffffffu, reject);
  const int k = rej ? (__ffs(rej) - 1) : gb;
  const float mt_k = row_m(k);
  const double st_k = row_s(k);
  const int kd = gb + 1 + (k < gb ? k : 0);
  const float md_k = row_m(kd);
  const double sd_k = row_s(kd);
  if (i <= G && i != k) P.out_tokens[(size_t)b * (G + 1) + i] = i < k ? x : -1;
  if (i < G) {
    const bool evaluated = i < gb && i <= k;
    if (P.p_tok) P.p_tok[(size_t)b * G + i] = evaluated ? p : NAN;
    if (P.q_tok) P.q_tok[(size_t)b * G + i] = evaluated ? q : NAN;
  }
  const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0) {
    P.num_accepted[b] = k;
    Decision d;
    d.k = k;
    d.reject = k < gb ? 1 : 0;
    d.mt = mt_k;
    d.md = d.reject ? md_k : 0.0f;
    d.inv_st = (float)(1.0 / st_k);
    d.rho = d.reject ? (float)(st_k / sd_k) : 0.0f;
    d.c_hi = tc.hi;
    d.c_lo = tc.lo;
    P.dec[b] = d;
    if (any) atomicOr(P.status, any);
    P.cnt_a[b] = 0;
    // publish the decision
    __threadfence();
    st_release(&P.ready[b], 1u);
  }
  __syncwarp();
}

// Greedy decision: argmax per target row from the per-item partials, then the
// first mismatch by warp ballot.
__device__ __noinline__ void decide_greedy(const Params& P, int b) {
  const int G = P.G, V = P.V, NC = P.NC;
  const int lane = threadIdx.x & 31;
  const int gb = clamp_gamma(P.gamma[b], G);
  unsigned int flags = (P.gamma[b] != gb) ? SV_STATUS_BAD_GAMMA : 0u;
  int g_mine = 0;  // lane r holds the argmax of row r
  for (int r = 0; r <= gb; ++r) {
    const float2* pr = P.stats + ((size_t)b * (2 * G + 1) + r) * P.stride_nc;
    float v = -INFINITY;
    int idx = 0x7fffffff;
    for (int c = lane; c < NC; c += 32) {
      const float2 mi = __ldcg(&pr[c]);
      argmax_combine(v, idx, mi.x, __float_as_int(mi.y));
    }
    warp_argmax(v, idx);
    if (!isfinite(v)) flags |= SV_STATUS_NONFINITE_ROW;
    if (lane == r) g_mine = (idx >= 0 && idx < V) ? idx : 0;
  }
  const int i = lane;
  int x = 0;
  bool mismatch = false;
  if (i < gb) {
    x = P.tokens[(size_t)b * G + i];
    if (x < 0 || x >= V) flags |= SV_STATUS_BAD_TOKEN;
    mismatch = x != g_mine;
  }
  const unsigned int mm = __ballot_sync(0xffffffffu, mismatch);
  const int k = mm ? (__ffs(mm) - 1) : gb;
  const int gk = __shfl_sync(0xffffffffu, g_mine, k);
  if (i <= G) P.out_tokens[(size_t)b * (G + 1) + i] = i < k ? x : (i == k ? gk : -1);
  const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0) {
    P.num_accepted[b] = k;
    if (any) atomicOr(P.status, any);
    P.cnt_a[b] = 0;
  }
  __syncwarp();
}

// Final draw for request b, run by the warp that completed its last R item:
// the chunk whose prefix passes u*S, then a scan of that chunk only.
template <int EB>
__device__ __noinline__ void final_draw(const Params& P, int b) {
  constexpr int RE = kHalfBytes / EB;  // elements per R chunk
  constexpr int EPL = RE / 32;         // contiguous elements per lane in the scan
  const int G = P.G, V = P.V, NCR = P.NCR;
  const int lane = threadIdx.x & 31;
  const Decision d = load_decision(&P.dec[b]);
  unsigned int flags = 0;
  const float u_s = sanitize_uniform(P.uniforms[(size_t)b * (G + 1) + G], flags);
  const ulonglong2* rp = P.resid + (size_t)b * P.stride_ncr;

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
  int cs = -1;
  for (int c0 = 0; c0 < NCR && cs < 0; c0 += 32) {
    const int c = c0 + lane;
    unsigned long long w = 0;
    if (c < NCR) {
      const ulonglong2 ww = __ldcg(&rp[c]);
      w = usep ? ww.y : ww.x;
    }
    const unsigned long long incl = warp_incl_scan_u64(w);
    const unsigned int hit = __ballot_sync(0xffffffffu, c < NCR && carry + incl > target);
    if (hit) {
      const int l = __ffs(hit) - 1;
      cs = c0 + l;
      base = carry + __shfl_sync(0xffffffffu, incl - w, l);
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  const int k = d.k < 0 ? 0 : (d.k > G ? G : d.k);
  int tok = -1;
  if (cs >= 0) {
    ResidC kc;
    kc.mt = d.mt; kc.md = d.md; kc.inv_st = d.inv_st; kc.rho = d.rho;
    kc.hi = d.c_hi; kc.lo = d.c_lo; kc.reject = (d.reject && k < G) ? 1 : 0;
    const char* trow = P.target + target_row(b, k, G, V) * EB;
    const char* drow = kc.reject ? P.draft + draft_row(b, k, G, V) * EB : nullptr;
    // This lane's EPL contiguous logits of the chosen chunk, one 16-byte
    // vector at a time (scalar loads when the rows do not allow it; -inf past
    // the end of the row).  Pass 1 sums the weights, pass 2 (one lane) finds
    // the token.
    constexpr int VEC = 16 / EB;
    constexpr int NV = EPL / VEC;
    const size_t e0 = (size_t)cs * RE + (size_t)lane * EPL;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(trow) |
                          reinterpret_cast<uintptr_t>(drow)) & 15) == 0 &&
                        e0 + EPL <= (size_t)V;
    auto load_vec = [&](const char* row, int q) -> uint4 {
      if (!row) return neg_inf_vec(EB);
      if (vec_ok) return __ldcg(reinterpret_cast<const uint4*>(row + (e0 + (size_t)q * VEC) * EB));
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (EB == 2) {
          const size_t ea = e0 + (size_t)q * 8 + 2 * h, eb = ea + 1;
          const uint32_t lo = ea < (size_t)V ? reinterpret_cast<const unsigned short*>(row)[ea] : 0xff80u;
          const uint32_t hi = eb < (size_t)V ? reinterpret_cast<const unsigned short*>(row)[eb] : 0xff80u;
          w[h] = lo | (hi << 16);
        } else {
          const size_t e = e0 + (size_t)q * 4 + h;
          w[h] = e < (size_t)V ? __float_as_uint(reinterpret_cast<const float*>(row)[e]) : 0xff800000u;
        }
      }
      return make_uint4(w[0], w[1], w[2], w[3]);
    };
    unsigned long long lsum = 0;
#pragma unroll 2
    for (int q = 0; q < NV; ++q) {
      const uint4 tv = load_vec(trow, q), dv = load_vec(drow, q);
#pragma unroll
      for (int h = 0; h < VEC; ++h) {
        unsigned long long wr, wp;
        resid_weights(vec_elem<EB>(tv, h), vec_elem<EB>(dv, h), kc, wr, wp);
        lsum += usep ? wp : wr;
      }
    }
    const unsigned long long incl = warp_incl_scan_u64(lsum);
    unsigned long long run = base + incl - lsum;
    if (run <= target && run + lsum > target) {
      for (int q = 0; q < NV && tok < 0; ++q) {
        const uint4 tv = load_vec(trow, q), dv = load_vec(drow, q);
#pragma unroll
        for (int h = 0; h < VEC; ++h) {
          unsigned long long wr, wp;
          resid_weights(vec_elem<EB>(tv, h), vec_elem<EB>(dv, h), kc, wr, wp);
          const unsigned long long nxt = run + (usep ? wp : wr);
          if (tok < 0 && nxt > target) tok = (int)(e0 + (size_t)(q * VEC + h));
          run = nxt;
        }
      }
    }
    const unsigned int own = __ballot_sync(0xffffffffu, tok >= 0);
    tok = own ? __shfl_sync(0xffffffffu, tok, __ffs(own) - 1) : -1;
  }
  if (lane == 0) {
    if (tok < 0) {
      flags |= SV_STATUS_INTERNAL;
      tok = V - 1;
    }
    P.out_tokens[(size_t)b * (G + 1) + k] = tok;
    if (flags) atomicOr(P.status, flags);
    P.cnt_r[b] = 0;
    P.ready[b] = 0;  // every R item of b is done: nobody reads the flag again
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Item processing (one warp per item)
// ---------------------------------------------------------------------------
// Element e of the item's row half h (0: p0, 1: p1) from global memory
// (unaligned items, which are not copied into the stage).
template <int EB>
__device__ __forceinline__ float direct_elem(const Meta& m, int h, int e) {
  return load_elem<EB>(h ? m.p1 : m.p0, (size_t)e);
}


// A item, sampling: (max, sum of exp2) over the item.
template <int EB>
__device__ __forceinline__ float2 a_item_sample(const Meta& m, const char* stage) {
  constexpr int VEC = 16 / EB;
  constexpr int NV = kItemBytes / 16 / 32;  // vectors per lane (16)
  const int lane = threadIdx.x & 31;
  float mx = -INFINITY, sum = 0.0f;
  if (!m.direct) {
    // two passes over the stage: the maximum, then the exponentials
    const int nvec = m.n / VEC;  // n * EB is a multiple of 16 on this path
    if constexpr (EB == 2) {
      // The item's 2*NV*4 logits stay in registers as bf16 pairs.
      constexpr int NW = NV * 4;
      uint32_t w[NW];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int vi = lane + 32 * j;
        const uint4 v = vi < nvec ? lds128(stage + vi * 16) : neg_inf_vec(EB);
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
      }
      // maximum on the packed pairs (exact), as a log-depth tree
      uint32_t t[NW / 2];
#pragma unroll
      for (int i = 0; i < NW / 2; ++i) t[i] = bf16x2_max(w[i], w[i + NW / 2]);
#pragma unroll
      for (int width = NW / 4; width >= 1; width >>= 1)
#pragma unroll
        for (int i = 0; i < width; ++i) t[i] = bf16x2_max(t[i], t[i + width]);
      mx = warp_max(bf16x2_hmax(t[0]));
      if (mx > -INFINITY) {
        // (z - m) * (hi + lo) and the sum, on float32 pairs, 8 accumulators
        const unsigned long long negm = f2_pack(-mx, -mx);
        const unsigned long long chi = f2_pack(m.c_hi, m.c_hi), clo = f2_pack(m.c_lo, m.c_lo);
        unsigned long long acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0ull;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
          const unsigned long long d = f2_add(bf16x2_to_f2(w[i]), negm);
          const unsigned long long a = f2_fma(d, chi, f2_mul(d, clo));
          float a0, a1;
          f2_unpack(a, a0, a1);
          acc[i & 7] = f2_add(acc[i & 7], f2_pack(ex2_approx(a0), ex2_approx(a1)));
        }
#pragma unroll
        for (int width = 4; width >= 1; width >>= 1)
#pragma unroll
          for (int i = 0; i < width; ++i) acc[i] = f2_add(acc[i], acc[i + width]);
        float s0, s1;
        f2_unpack(acc[0], s0, s1);
        sum = s0 + s1;
      }
      return make_float2(mx, warp_sum(sum));
    }
    uint4 v[NV];  // float32: the item stays in registers
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vi = lane + 32 * j;
      v[j] = vi < nvec ? lds128(stage + vi * 16) : neg_inf_vec(EB);
    }
    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
      for (int q = 0; q < VEC; ++q) mq[q & 3] = fmaxf(mq[q & 3], vec_elem<EB>(v[j], q));
    mx = warp_max(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])));
    if (mx > -INFINITY) {
      float sq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        float e[VEC];
#pragma unroll
        for (int q = 0; q < VEC; ++q)
          e[q] = ex2_approx(exp_arg(vec_elem<EB>(v[j], q), mx, m.c_hi, m.c_lo));
#pragma unroll
        for (int w = VEC; w > 1; w >>= 1)
#pragma unroll
          for (int q = 0; q < w / 2; ++q) e[q] = e[2 * q] + e[2 * q + 1];
        sq[j & 3] += e[0];
      }
      sum = (sq[0] + sq[1]) + (sq[2] + sq[3]);
    }
  } else {
    for (int e = lane; e < m.n; e += 32) mx = fmaxf(mx, direct_elem<EB>(m, 0, e));
    mx = warp_max(mx);
    if (mx > -INFINITY)
      for (int e = lane; e < m.n; e += 32)
        sum += ex2_approx(exp_arg(direct_elem<EB>(m, 0, e), mx, m.c_hi, m.c_lo));
  }
  sum = warp_sum(sum);
  return make_float2(mx, sum);
}

// A item, greedy: (max, lowest row-global index of the max).
template <int EB>
__device__ __forceinline__ float2 a_item_greedy(const Meta& m, const char* stage) {
  constexpr int VEC = 16 / EB;
  constexpr int NV = kItemBytes / 16 / 32;
  constexpr int AE = kItemBytes / EB;
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  if (!m.direct) {
    // the maximum (independent chains), then the lowest index holding it
    const int nvec = m.n / VEC;
    if constexpr (EB == 2) {
      // maximum on the packed pairs as a log-depth tree; a lane holding the
      // warp maximum finds its first vector holding it, then the element
      constexpr int NW = NV * 4;
      uint32_t w[NW];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int vi = lane + 32 * j;
        const uint4 v = vi < nvec ? lds128(stage + vi * 16) : neg_inf_vec(EB);
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
      }
      uint32_t t[NW / 2];
#pragma unroll
      for (int i = 0; i < NW / 2; ++i) t[i] = bf16x2_max(w[i], w[i + NW / 2]);
#pragma unroll
      for (int width = NW / 4; width >= 1; width >>= 1)
#pragma unroll
        for (int i = 0; i < width; ++i) t[i] = bf16x2_max(t[i], t[i + width]);
      const float lm = bf16x2_hmax(t[0]);
      bv = warp_max(lm);
      unsigned int idx = 0x7fffffffu;
      if (lm == bv) {
        const uint32_t b16 = __float_as_uint(bv) >> 16;
        const uint32_t b2 = b16 | (b16 << 16);
        unsigned int mask = 0;  // bit j: vector j holds the maximum
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          const uint32_t e = bf16x2_eq(w[4 * j], b2) | bf16x2_eq(w[4 * j + 1], b2) |
                             bf16x2_eq(w[4 * j + 2], b2) | bf16x2_eq(w[4 * j + 3], b2);
          mask |= (e != 0u ? 1u : 0u) << j;
        }
        if (mask) {
          const int j = __ffs(mask) - 1;
          const int vi = lane + 32 * j;
          const uint4 v = lds128(stage + vi * 16);
#pragma unroll
          for (int q = VEC - 1; q >= 0; --q)
            if (vec_elem<EB>(v, q) == bv) idx = (unsigned int)(vi * VEC + q);
        }
      }
      bi = (int)__reduce_min_sync(0xffffffffu, idx);
      return make_float2(bv, __int_as_float(bi == 0x7fffffff ? bi : m.c * AE + bi));
    }
    uint4 v[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vi = lane + 32 * j;
      v[j] = vi < nvec ? lds128(stage + vi * 16) : neg_inf_vec(EB);
    }
    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
      for (int q = 0; q < VEC; ++q) mq[q & 3] = fmaxf(mq[q & 3], vec_elem<EB>(v[j], q));
    bv = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
    // this lane's elements in increasing index order: vector j, element q
#pragma unroll
    for (int j = NV - 1; j >= 0; --j)
#pragma unroll
      for (int q = VEC - 1; q >= 0; --q) {
        const int vi = lane + 32 * j;
        if (vi < nvec && vec_elem<EB>(v[j], q) == bv) bi = vi * VEC + q;
      }
  } else {
    for (int e = lane; e < m.n; e += 32) argmax_combine(bv, bi, direct_elem<EB>(m, 0, e), e);
  }
  warp_argmax(bv, bi);
  return make_float2(bv, __int_as_float(bi == 0x7fffffff ? bi : m.c * AE + bi));
}

// R item: fixed-point sums of the residual weights and of p over the chunk.
template <int EB>
__device__ __forceinline__ ulonglong2 r_item(const Meta& m, const char* stage) {
  constexpr int VEC = 16 / EB;
  constexpr int NV = kHalfBytes / 16 / 32;  // vectors per lane per row (8)
  const int lane = threadIdx.x & 31;
  ResidC kc;
  kc.mt = m.mt; kc.md = m.md; kc.inv_st = m.inv_st; kc.rho = m.rho;
  kc.hi = m.c_hi; kc.lo = m.c_lo; kc.reject = m.reject;
  unsigned long long sr = 0, sp = 0;
  if (!m.direct) {
    const int nvec = m.n / VEC;
    unsigned long long ar[2] = {0, 0}, ap[2] = {0, 0};  // independent chains
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vi = lane + 32 * j;
      if (vi < nvec) {
        const uint4 t = lds128(stage + vi * 16);
        const uint4 d = m.reject ? lds128(stage + kHalfBytes + vi * 16) : neg_inf_vec(EB);
#pragma unroll
        for (int q = 0; q < VEC; ++q) {
          unsigned long long wr, wp;
          resid_weights(vec_elem<EB>(t, q), vec_elem<EB>(d, q), kc, wr, wp);
          ar[q & 1] += wr;
          ap[q & 1] += wp;
        }
      }
    }
    sr = ar[0] + ar[1];
    sp = ap[0] + ap[1];
  } else {
    for (int e = lane; e < m.n; e += 32) {
      unsigned long long wr, wp;
      const float zd = m.reject ? direct_elem<EB>(m, 1, e) : -INFINITY;
      resid_weights(direct_elem<EB>(m, 0, e), zd, kc, wr, wp);
      sr += wr;
      sp += wp;
    }
  }
  return make_ulonglong2(warp_sum_u64(sr), warp_sum_u64(sp));
}

// ---------------------------------------------------------------------------
// Work items: one fixed order, claimed in small batches
// ---------------------------------------------------------------------------
// First the A items of every request (request-major: rows, then chunks), then
// the R items of every request.  The R tail starts D requests before the end
// and walks backwards (wrapping to the last D at the very end): the first R
// items re-read the most recently streamed rows, which are still in L2, while
// the last D requests, decided last, come last.  A warp walks its batch with
// a cursor that advances in O(1) per item.
struct Cursor {
  unsigned int j;   // item index
  int req, row, c;  // A: request, row within the request, chunk
  int rows, gb;     // A: rows of req, and its gamma
  int rank;         // R: position in the tail
};

template <int MODE>
__device__ __forceinline__ int rows_of(const int* rowpre, int b) {
  return rowpre[b + 1] - rowpre[b];
}

// Place the cursor on item j.
template <int MODE>
__device__ __forceinline__ void cursor_seek(Cursor& k, unsigned int j, const int* rowpre, int B,
                                            int NC, int NCR, unsigned int nA) {
  k.j = j;
  if (MODE == MODE_SAMPLE && j >= nA) {
    k.rank = (int)((j - nA) / NCR);
    k.c = (int)((j - nA) % NCR);
    return;
  }
  int lo = 0, hi = B - 1;  // largest request with rowpre[b] * NC <= j
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((unsigned int)rowpre[mid] * NC <= j) lo = mid; else hi = mid - 1;
  }
  const unsigned int off = j - (unsigned int)rowpre[lo] * NC;
  k.req = lo;
  k.row = (int)(off / NC);
  k.c = (int)(off % NC);
  k.rows = rows_of<MODE>(rowpre, lo);
  k.gb = MODE == MODE_SAMPLE ? (k.rows - 1) / 2 : k.rows - 1;
}

// Advance the cursor by one item.
template <int MODE>
__device__ __forceinline__ void cursor_next(Cursor& k, const int* rowpre, int NC, int NCR,
                                            unsigned int nA) {
  ++k.j;
  if (MODE == MODE_SAMPLE && k.j > nA) {  // inside the R tail
    if (++k.c == NCR) {
      k.c = 0;
      ++k.rank;
    }
    return;
  }
  if (MODE == MODE_SAMPLE && k.j == nA) {  // first R item
    k.rank = 0;
    k.c = 0;
    return;
  }
  if (++k.c == NC) {
    k.c = 0;
    if (++k.row == k.rows) {
      k.row = 0;
      ++k.req;
      k.rows = rows_of<MODE>(rowpre, k.req);
      k.gb = MODE == MODE_SAMPLE ? (k.rows - 1) / 2 : k.rows - 1;
    }
  }
}

// The A item under the cursor.
template <int EB, int MODE>
__device__ __forceinline__ void a_item_at(const Params& P, const Cursor& k, float c_hi,
                                          float c_lo, Meta& m) {
  constexpr int AE = kItemBytes / EB;
  const int G = P.G, V = P.V;
  size_t roff;
  const char* base;
  if (k.row <= k.gb) {
    m.pslot = k.row;
    roff = target_row(k.req, k.row, G, V);
    base = P.target;
  } else {
    const int i = k.row - k.gb - 1;
    m.pslot = G + 1 + i;
    roff = draft_row(k.req, i, G, V);
    base = P.draft;
  }
  m.kind = KIND_A;
  m.b = k.req;
  m.c = k.c;
  m.n = min(AE, V - k.c * AE);
  m.p0 = base + (roff + (size_t)k.c * AE) * EB;
  m.p1 = nullptr;
  m.direct = (((reinterpret_cast<uintptr_t>(m.p0)) & 15) != 0 || ((m.n * EB) & 15) != 0) ? 1 : 0;
  m.c_hi = c_hi;
  m.c_lo = c_lo;
}

// Complete R item m (request m.b, chunk m.c) from its request's decision.
template <int EB>
__device__ __forceinline__ void fill_r_item(const Params& P, const Decision& d, Meta& m) {
  constexpr int RE = kHalfBytes / EB;
  const int G = P.G, V = P.V, req = m.b, c = m.c;
  const int k = d.k < 0 ? 0 : (d.k > G ? G : d.k);
  const int reject = (d.reject && k < G) ? 1 : 0;
  m.kind = KIND_R;
  m.pslot = k;
  m.reject = reject;
  m.n = min(RE, V - c * RE);
  m.p0 = P.target + (target_row(req, k, G, V) + (size_t)c * RE) * EB;
  m.p1 = reject ? P.draft + (draft_row(req, k, G, V) + (size_t)c * RE) * EB : nullptr;
  const uintptr_t a = reinterpret_cast<uintptr_t>(m.p0) | reinterpret_cast<uintptr_t>(m.p1);
  m.direct = ((a & 15) != 0 || ((m.n * EB) & 15) != 0) ? 1 : 0;
  m.mt = d.mt;
  m.md = d.md;
  m.inv_st = d.inv_st;
  m.rho = d.rho;
  m.c_hi = d.c_hi;
  m.c_lo = d.c_lo;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int EB, int MODE>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(Params P) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  int* rowpre = reinterpret_cast<int*>(dsmem + kWarps * kNB * kItemBytes);  // [B+1]
  __shared__ __align__(8) uint64_t bar[kWarps][kNB];
  __shared__ Meta meta[kWarps][kNB];     // the item in each buffer
  __shared__ int2 defq[kWarps][kDefer];  // deferred R items (request, chunk)
  __shared__ int sh_carry;
  __shared__ int wsum[kWarps];
  __shared__ int sh_last;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = P.G, B = P.B, NC = P.NC;
  const int NCR = MODE == MODE_SAMPLE ? P.NCR : 1;

  if (tid == 0) {
    rowpre[0] = 0;
    sh_carry = 0;
    for (int w = 0; w < kWarps; ++w)
      for (int s = 0; s < kNB; ++s) mbar_init(&bar[w][s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // rows per request -> exclusive prefix in shared memory
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + tid;
    int v = 0;
    if (b < B) {
      const int gb = clamp_gamma(P.gamma[b], G);
      v = MODE == MODE_SAMPLE ? 2 * gb + 1 : gb + 1;
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int off = sh_carry;
    for (int w = 0; w < warp; ++w) off += wsum[w];
    if (b < B) rowpre[b + 1] = off + incl;
    __syncthreads();
    if (tid == kThreads - 1) sh_carry = off + incl;
    __syncthreads();
  }

  const unsigned int nA = (unsigned int)rowpre[B] * NC;
  const unsigned int total = nA + (MODE == MODE_SAMPLE ? (unsigned int)B * NCR : 0u);
  const unsigned int nwarps = gridDim.x * kWarps;
  // batches: about 1/kBatchDiv of a warp's share, at most kMaxK items
  const unsigned int K = min((unsigned int)kMaxK, max(1u, total / (nwarps * kBatchDiv)));
  int D = 1;  // requests whose A items may still be in flight when the tail starts
  {
    const double per_req = (double)nA / (double)(B > 0 ? B : 1);
    D = (int)ceil((double)nwarps * (kNB + K) / per_req) + 1;
    D = D < B ? D : B - 1;
  }

  unsigned char* mybuf = dsmem + (size_t)warp * kNB * kItemBytes;
  uint64_t* mybar = bar[warp];
  Meta* mymeta = meta[warp];
  int2* mydef = defq[warp];

  unsigned int nb = 0;  // lane 0: start of the pre-claimed next batch
  if (lane == 0) nb = atomicAdd(P.next_item, K);

  Cursor cur;
  cur.j = 0;
  unsigned int cur_end = 0;  // the current batch is [cur.j, cur_end)
  int a_tb = -1;             // request whose temperature constants are in a_hi/a_lo
  float a_hi = 0.0f, a_lo = 0.0f;
  bool more = true;          // batches may remain
  unsigned int issued = 0, processed = 0;
  int dec_b = -1;            // request whose decision is in dc (warp-uniform)
  Decision dc;
  dc.k = 0;
  int defhead = 0, ndef = 0;  // ring of deferred R items (warp-uniform)
  bool blocked = false;       // waiting for the oldest deferred item's decision
  int acc_kind = KIND_A, acc_b = 0;
  unsigned int acc_n = 0;     // arrivals held for (acc_kind, acc_b)
  unsigned int flags = 0;
  bool failed = false;

  // Arrivals are published asynchronously: flush() adds the held count with
  // one acquire-release atomic; its result is examined at the next settle(),
  // and the warp that completed a request then runs the request's follow-up.
  unsigned int pend_old = 0, pend_n = 0, pend_total = 0;  // lane 0
  int pend_kind = KIND_A, pend_b = -1;                      // warp-uniform
  auto settle = [&]() {
    if (pend_b < 0) return;
    unsigned int last = 0;
    if (lane == 0) last = (pend_old + pend_n == pend_total) ? 1u : 0u;
    last = __shfl_sync(0xffffffffu, last, 0);
    const int b = pend_b;
    pend_b = -1;
    if (last) {
      if (pend_kind == KIND_A) {
        if (MODE == MODE_SAMPLE) decide_sample<EB>(P, b);
        else decide_greedy(P, b);
      } else {
        final_draw<EB>(P, b);
      }
    }
  };
  auto flush = [&]() {
    if (acc_n == 0) return;
    settle();
    if (lane == 0) {
      unsigned int* cnt = acc_kind == KIND_A ? &P.cnt_a[acc_b] : &P.cnt_r[acc_b];
      pend_total = acc_kind == KIND_A ? (unsigned int)rows_of<MODE>(rowpre, acc_b) * (unsigned int)NC
                                      : (unsigned int)NCR;
      pend_n = acc_n;
      pend_old = atom_add_acq_rel(cnt, acc_n);
    }
    pend_kind = acc_kind;
    pend_b = acc_b;
    acc_n = 0;
  };

  // Is request b decided?  If so its decision is fetched into dc.
  auto decided = [&](int b) -> bool {
    if (b == dec_b) return true;
    unsigned int ok = 0;
    Decision d;
    d.k = 0;
    if (lane == 0 && ld_acquire(&P.ready[b])) {
      ok = 1;
      d = load_decision(&P.dec[b]);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      dc.k = __shfl_sync(0xffffffffu, d.k, 0);
      dc.reject = __shfl_sync(0xffffffffu, d.reject, 0);
      dc.mt = __shfl_sync(0xffffffffu, d.mt, 0);
      dc.md = __shfl_sync(0xffffffffu, d.md, 0);
      dc.inv_st = __shfl_sync(0xffffffffu, d.inv_st, 0);
      dc.rho = __shfl_sync(0xffffffffu, d.rho, 0);
      dc.c_hi = __shfl_sync(0xffffffffu, d.c_hi, 0);
      dc.c_lo = __shfl_sync(0xffffffffu, d.c_lo, 0);
      dec_b = b;
    }
    return ok != 0;
  };

  // Start the copy of item m into the next buffer (lane 0).
  auto issue = [&](const Meta& m) {
    const int s = (int)(issued % kNB);
    if (lane == 0) {
      mymeta[s] = m;
      unsigned char* dst = mybuf + s * kItemBytes;
      // The buffer's previous item was fully read: its values were consumed by
      // the reductions before the __syncwarp that ended its processing.
      if (m.direct) {
        mbar_arrive(&mybar[s]);
      } else {
        const unsigned int bytes = (unsigned int)(m.n * EB);
        const bool two = m.kind == KIND_R && m.p1 != nullptr;
        mbar_arrive_expect_tx(&mybar[s], two ? 2 * bytes : bytes);
        bulk_copy_g2s(dst, m.p0, bytes, &mybar[s]);
        if (two) bulk_copy_g2s(dst + kHalfBytes, m.p1, bytes, &mybar[s]);
      }
    }
    __syncwarp();
    ++issued;
  };

  while (!failed) {
    // 1. keep kNB copies in flight
    while (!blocked && issued - processed < (unsigned int)kNB) {
      if (cur.j == cur_end) {
        // batch boundary: first the oldest deferred R item, if now decided
        if (MODE == MODE_SAMPLE && ndef > 0 && decided(mydef[defhead].x)) {
          Meta r;
          r.b = mydef[defhead].x;
          r.c = mydef[defhead].y;
          fill_r_item<EB>(P, dc, r);
          issue(r);
          defhead = (defhead + 1) % kDefer;
          --ndef;
          continue;
        }
        if (more) {
          const unsigned int base = __shfl_sync(0xffffffffu, nb, 0);
          if (base >= total) {
            more = false;
          } else {
            cursor_seek<MODE>(cur, base, rowpre, B, NC, NCR, nA);
            cur_end = min(base + K, total);
            if (lane == 0) nb = atomicAdd(P.next_item, K);  // pre-claim the next batch
          }
        }
        if (cur.j == cur_end) {
          if (ndef > 0) blocked = true;  // only deferred items remain
          break;
        }
      }
      if (MODE == MODE_SAMPLE && cur.j >= nA) {
        // R item: its request's rows depend on the decision
        Meta r;
        r.b = (2 * B - 1 - D - cur.rank) % B;
        r.c = cur.c;
        if (decided(r.b)) {
          fill_r_item<EB>(P, dc, r);
          issue(r);
        } else {
          // not decided yet: set it aside and keep streaming later items
          if (ndef == kDefer) {
            blocked = true;
            break;
          }
          if (lane == 0) mydef[(defhead + ndef) % kDefer] = make_int2(r.b, r.c);
          __syncwarp();
          ++ndef;
        }
      } else {
        if (MODE == MODE_SAMPLE && cur.req != a_tb) {
          unsigned int fl = 0;
          const TempC tc = temp_consts(sanitize_temperature(P.temperature[cur.req], fl));
          a_hi = tc.hi;
          a_lo = tc.lo;
          a_tb = cur.req;
        }
        Meta a;
        a_item_at<EB, MODE>(P, cur, a_hi, a_lo, a);
        issue(a);
      }
      cursor_next<MODE>(cur, rowpre, NC, NCR, nA);
    }

    // 2. process the oldest item in flight
    if (issued != processed) {
      const int s = (int)(processed % kNB);
      if (!mbar_wait(&mybar[s], (processed / kNB) & 1u)) {
        flags |= SV_STATUS_TIMEOUT;
        failed = true;
        break;
      }
      const Meta& m = mymeta[s];
      const int m_kind = m.kind, m_b = m.b;
      const char* stage = reinterpret_cast<const char*>(mybuf + s * kItemBytes);
      if (m_kind == KIND_A) {
        const float2 part = MODE == MODE_SAMPLE ? a_item_sample<EB>(m, stage)
                                                : a_item_greedy<EB>(m, stage);
        if (lane == 0) P.stats[((size_t)m_b * (2 * G + 1) + m.pslot) * P.stride_nc + m.c] = part;
      } else {
        const ulonglong2 part = r_item<EB>(m, stage);
        if (lane == 0) P.resid[(size_t)m_b * P.stride_ncr + m.c] = part;
      }
      __syncwarp();  // every lane is done with the buffer before it is reused
      ++processed;
      settle();
      if (acc_n && (m_kind != acc_kind || m_b != acc_b)) flush();
      acc_kind = m_kind;
      acc_b = m_b;
      ++acc_n;
      continue;
    }

    // 3. nothing in flight
    if (blocked) {
      // Publish held arrivals, then wait for the oldest deferred item's
      // request.  Everything this warp still holds is either a deferred R item
      // (no decision depends on one) or comes later in the order.
      flush();
      settle();
      int state = 0;
      if (lane == 0) {
        const unsigned long long t0 = now_ns();
        while (!ld_acquire(&P.ready[mydef[defhead].x])) {
          if (now_ns() - t0 > kWaitNs) {
            state = 1;
            break;
          }
          __nanosleep(128);
        }
      }
      if (__shfl_sync(0xffffffffu, state, 0)) {
        flags |= SV_STATUS_TIMEOUT;
        failed = true;
        break;
      }
      blocked = false;
      continue;
    }
    if (!more && cur.j == cur_end && ndef == 0) break;  // all work done
  }

  // No copy may still be landing in this warp's buffers when it leaves.
  if (failed) {
    for (unsigned int p = processed; p < issued; ++p)
      (void)mbar_wait(&mybar[p % kNB], (p / kNB) & 1u);
  } else {
    flush();
    settle();
  }
  if (lane == 0 && flags) atomicOr(P.status, flags);
  __syncthreads();
  // the last CTA out resets the claim counter for the next call
  if (tid == 0) {
    __threadfence();
    sh_last = atomicAdd(P.exit_count, 1u) == gridDim.x - 1 ? 1 : 0;
    if (sh_last) {
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

constexpr size_t kMaxSmem =
    (size_t)kWarps * kNB * kItemBytes + (size_t)(kMaxBatch + 1) * sizeof(int);

// Persistent grid: as many CTAs as fit on the device (cached per device).
template <int EB, int MODE>
int grid_size() {
  static int cached_dev = -1, cached_grid = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev == cached_dev && cached_grid > 0) return cached_grid;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(verify_kernel<EB, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kMaxSmem) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<EB, MODE>, kThreads,
                                                    kMaxSmem) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_grid = sms * (per_sm > 0 ? per_sm : 1);
  return cached_grid;
}

template <int EB, int MODE>
int launch(const Params& P, cudaStream_t stream) {
  const int grid = grid_size<EB, MODE>();
  if (grid <= 0) return SV_ERR_CUDA;
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
    Q.stats = P.stats + (size_t)b0 * (2 * G + 1) * P.stride_nc;
    Q.resid = P.resid + (size_t)b0 * P.stride_ncr;
    const size_t smem = (size_t)kWarps * kNB * kItemBytes + (size_t)(Q.B + 1) * sizeof(int);
    verify_kernel<EB, MODE><<<grid, kThreads, smem, stream>>>(Q);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  }
  return SV_OK;
}

int fill_params(Params& P, const void* target, const void* draft, sv_dtype dtype, int B, int G,
                int V, const int32_t* tokens, const int32_t* gamma, const float* uniforms,
                const float* temperature, int32_t* out_tokens, int32_t* num_accepted,
                double* p_tok, double* q_tok, void* ws, size_t ws_bytes) {
  const Layout L = make_layout(B, G, V);
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
  P.NC = (int)((V + kItemBytes / eb - 1) / (kItemBytes / eb));
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

// Scratch for spec_verify_sample_noalloc: part of the library's device
// image, so using it allocates nothing.  Its device address is looked up once
// per device.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

static __device__ __align__(256) unsigned char sv_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

namespace {

int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, sv_noalloc_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
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
  rc = fill_params(P, target_logits, draft_logits, dtype, B, G, V, draft_tokens, gamma, uniforms,
                   temperature, out_tokens, num_accepted, p_tok, q_tok, workspace, ws_bytes);
  if (rc) return rc;
  if (B == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == SV_BF16 ? launch<2, MODE_SAMPLE>(P, s) : launch<4, MODE_SAMPLE>(P, s);
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
  rc = fill_params(P, target_logits, nullptr, dtype, B, G, V, draft_tokens, gamma, nullptr,
                   nullptr, out_tokens, num_accepted, nullptr, nullptr, workspace, ws_bytes);
  if (rc) return rc;
  if (B == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == SV_BF16 ? launch<2, MODE_GREEDY>(P, s) : launch<4, MODE_GREEDY>(P, s);
}

int spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                               sv_dtype dtype, int B, int G, int V,
                               const int32_t* draft_tokens, const int32_t* gamma,
                               const float* uniforms, const float* temperature,
                               int32_t* out_tokens, int32_t* num_accepted, double* p_tok,
                               double* q_tok, sv_stream_t stream) {
  int rc = check_scalars(dtype, B, G, V);
  if (rc) return rc;
  if (!target_logits || !gamma || !uniforms || !temperature || !out_tokens || !num_accepted)
    return SV_ERR_NULL;
  if (G > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_NULL;
  const Layout L = make_layout(B, G, V);
  if (L.total > (size_t)SV_NOALLOC_SCRATCH_BYTES) return SV_ERR_STATIC_LIMIT;
  if (B == 0) return SV_OK;
  void* ws = nullptr;
  rc = noalloc_scratch(&ws);
  if (rc) return rc;
  Params P;
  rc = fill_params(P, target_logits, draft_logits, dtype, B, G, V, draft_tokens, gamma, uniforms,
                   temperature, out_tokens, num_accepted, p_tok, q_tok, ws,
                   (size_t)SV_NOALLOC_SCRATCH_BYTES);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // counters, arrival counts and decision flags start at zero for every call
  if (cudaMemsetAsync(ws, 0, L.dec, s) != cudaSuccess) return SV_ERR_CUDA;
  return dtype == SV_BF16 ? launch<2, MODE_SAMPLE>(P, s) : launch<4, MODE_SAMPLE>(P, s);
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
    case SV_ERR_STATIC_LIMIT: return "sizes need more scratch than the built-in 4 MiB array";
    default: return "unknown error code";
  }
}

}  // extern "C"
