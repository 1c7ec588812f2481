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
// A request whose temperature is 0 inside a sampling call takes the greedy
// steps.  Inputs come padded ([B][G+1] target rows, [B][G] draft rows) or
// packed (rows back to back, addressed through a prefix of the draft
// lengths); a draft-token sampler (G = 0, no drafts) shares the same kernel.
//
// Each call is one launch of one of three kernels (the choice: `route`, near
// the end of this file):
//   cluster_kernel  small batches: one thread-block cluster per request whose
//                   warps each hold one chunk of a position's target and draft
//                   rows; partials, decision and residual stay in the
//                   cluster's shared memory (section "Small batches" below);
//   stream_kernel   up to one cluster per SM: the request's chunks streamed by
//                   its cluster; beyond that, CTAs claiming whole requests in
//                   turn, longest first (section "Medium batches");
//   verify_kernel   the persistent grid described next, for batches whose
//                   claim order does not fit in shared memory.
// All three reduce items with the same routines and decide and draw with the
// same code, so their outputs agree bit for bit.
//
// The persistent grid: one CTA of 12 warps per SM.  Work items:
//   A items  8 KB of one logit row -> (max, sum of exp2((z - max) log2(e)/T))
//            when sampling, (max, lowest index of the max) when greedy.  All
//            A items of the batch come first, request-major: the first batch
//            of every warp is static, later batches are claimed from a
//            global counter ahead of use.
//   R items  4 KB of target row k and the same 4 KB of draft row k of one
//            rejecting request -> a 64-bit fixed-point sum of the residual
//            weights max(0, p_k - q_k) over the item.  They are claimed only
//            once the A items are all claimed.
// Every warp keeps two items in flight in private shared-memory buffers,
// filled by bulk copies (cp.async.bulk) and tracked by mbarriers; an item
// whose bytes are not 16-byte aligned is read with plain loads into its
// buffer instead, so both kinds are reduced by the same code.  Arrivals are
// counted per request (one release atomic per run of items of one request).
// The warp whose arrival completes a request's A items runs its decision on
// the spot: row statistics in float-float, the acceptance ratios, a ballot
// for the first reject; with every draft accepted it also draws the bonus
// token from the A statistics of target row gamma_b.  A reject is published
// to a queue of decision records; the warp whose arrival completes that
// request's R items locates the chunk holding u S and walks only that chunk
// for the token.  No warp waits for work that is not already claimed, every
// wait is bounded (2 s of global time) and ends in SV_STATUS_TIMEOUT, and
// counters are reset by their last user, so the workspace stays zeroed.
//
// Numerics: inputs widen exactly to float32.  Exponent arguments use a
// two-term log2(e)/T; exp2 is the SFU's ex2.approx.  Row sums combine item
// partials in float-float; the acceptance ratio 2^(e_t - e_d) S_d / S_t is
// formed from float-float exponents and an exp2 of the fractional part, with
// float64 only where an exponent is extreme and for the optional p/q outputs.
// Residual weights are summed in exact fixed point (units of 2^-39 of S_t),
// so chunk sums and the final in-chunk walk agree bit for bit and do not
// depend on summation order.

#include <cuda_runtime.h>
#include <atomic>
#include <mutex>
#include <stdint.h>
#include <math.h>
#include <float.h>

#include "spec_verify.h"

namespace {

#ifndef SV_WARPS
#define SV_WARPS 12
#endif
#ifndef SV_BACKLOG_X4
#define SV_BACKLOG_X4 64u  // R backlog, in quarter-batches per warp
#endif
#ifndef SV_BUFFERS
#define SV_BUFFERS 2
#endif
constexpr int kWarps = SV_WARPS;                      // warps per CTA (one CTA per SM)
constexpr int kThreads = 32 * kWarps;
constexpr int kNB = SV_BUFFERS;                       // TMA buffers per warp
constexpr int kItemBytes = 8192;                      // A item: 8 KB of one row
constexpr int kHalfBytes = kItemBytes / 2;            // R item: 4 KB of each of two rows
constexpr int kMaxBatch = 1536;                       // requests per launch (smem tables)
#ifndef SV_MAXK
#define SV_MAXK 8
#endif
constexpr int kMaxK = SV_MAXK;                        // A items per claimed batch
#ifndef SV_RUNROLL
#define SV_RUNROLL 2
#endif
constexpr int kRUnroll = SV_RUNROLL;                  // vector columns per step of an R item
#ifndef SV_MAXKR
#define SV_MAXKR 4u
#endif
constexpr unsigned int kMaxRBatch = SV_MAXKR;         // R items per claim, at most
#ifndef SV_BATCH_DIV
#define SV_BATCH_DIV 1u
#endif
// batches per warp's share of the A items, at least (a sweep over 1, 2 and 4
// on B = 64..512 found the largest batches best: claims cost more than
// the longer hold of the last requests' items)
constexpr unsigned int kBatchDiv = SV_BATCH_DIV;
constexpr unsigned long long kWaitNs = 2000000000ull; // default wait limit: 2 s
#ifndef SV_LAZY
#define SV_LAZY 1
#endif
// default of spec_verify_set_lazy: request claims test a sampled request's
// positions one at a time, reading a position's rows only when every earlier
// draft was accepted
constexpr int kLazyDefault = SV_LAZY != 0 ? 1 : 0;
#ifndef SV_SPEC_MIN_GAMMA
#define SV_SPEC_MIN_GAMMA 4
#endif
// A lazy request with at least this many drafts has its next position's rows
// read while a position is decided (the bonus row is not read ahead).  Short
// requests do not: for them the rows read ahead after a rejection cost more
// than the wait saved after an acceptance (B = 512: gamma 3, 174 against 178 us;
// ragged gamma 1..7: 135 against 132 us).
constexpr int kSpecMinGamma = SV_SPEC_MIN_GAMMA;

constexpr float kLog2eHi = 1.44269502162933349609375f;      // float nearest log2(e)
constexpr float kLog2eLo = 1.925963033500011e-08f;          // log2(e) - kLog2eHi

enum { KIND_A = 0, KIND_R = 1 };
enum { MODE_SAMPLE = 0, MODE_GREEDY = 1 };

// ---------------------------------------------------------------------------
// Workspace
// ---------------------------------------------------------------------------
// Per-request decision.
struct Decision {
  int k;               // first rejected position (gamma_b if none)
  int reject;          // 1: residual at k; 0: bonus from target row k = gamma_b
  float mt, md;        // maxima of target row k and draft row k
  float inv_st, rho;   // 1/S_t and S_t/S_d of those rows (from float-float sums)
  float c_hi, c_lo;    // log2(e)/T as hi + lo
};
// A published decision in the workspace: two 16-byte halves, each written and
// read with one 128-bit atomic and each carrying the tag kDecTag | reject << 8
// | k, so a reader that finds both tags set holds a consistent record without
// further ordering.  The same record serves as a request's own entry and as
// an entry of the decision queue (which also names the request).
constexpr uint32_t kDecTag = 0x80000000u;
struct __align__(16) DecRecord {
  uint32_t tag_a; int b; float mt, md;
  uint32_t tag_b; float inv_st, rho; uint32_t pad;
};

struct Layout {
  size_t status, next_item, exit_count, r_next, q_tail, dec_count;  // header words
  size_t cnt_a, cnt_r, dec, queue, stats, resid, total;
  int NC, NCR;  // worst-case chunk counts (float32 logits)
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline Layout make_layout(int B, int G, int V) {
  Layout L;
  L.NC = (V + kItemBytes / 4 - 1) / (kItemBytes / 4);
  L.NCR = (V + kHalfBytes / 4 - 1) / (kHalfBytes / 4);
  // header words on separate 128-byte lines
  L.status = 0;
  L.next_item = 128;
  L.exit_count = 256;
  L.r_next = 384;
  L.q_tail = 512;
  L.dec_count = 640;
  size_t off = 1024;
  L.cnt_a = off; off = align256(off + (size_t)B * 4);
  L.cnt_r = off; off = align256(off + (size_t)B * 4);
  L.dec = off;   off = align256(off + (size_t)B * sizeof(DecRecord));
  L.queue = off; off = align256(off + (size_t)B * sizeof(DecRecord));
  L.stats = off; off = align256(off + (size_t)B * (2 * G + 1) * L.NC * sizeof(float2));
  L.resid = off; off = align256(off + (size_t)B * L.NCR * sizeof(unsigned long long));
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
  const int32_t* cu;          // packed layout: [B+1] draft prefix (nullptr: padded layout)
  int total;                  // packed layout: drafts in all requests (rows of draft_logits)
  int b_base;                 // packed layout: global index of this launch's first request
  const float* uniforms;
  const float* temperature;
  int32_t* out_tokens;
  int32_t* num_accepted;
  double* p_tok;
  double* q_tok;
  unsigned int* status;
  unsigned long long wait_ns;  // every bounded wait gives up after this long
  int lazy;                   // request claims: positions one stage at a time
  unsigned int* next_item;   // next A item to claim (past the fixed first batches)
  unsigned int* r_next;      // next R item to claim: item i is chunk i % NCR of the
                             // request in queue slot i / NCR
  unsigned int* q_tail;      // decisions published to the queue (rejections only)
  unsigned int* dec_count;   // requests decided (written after any queue entry)
  unsigned int* exit_count;
  unsigned int* cnt_a;       // [B] A items completed
  unsigned int* cnt_r;       // [B] R items completed
  DecRecord* dec;            // [B] decision of each request (tags 0 until decided)
  DecRecord* queue;          // [B] decisions in the order they were made
  float2* stats;              // [B][2G+1][stride_nc]: (max, sum) or (max, argmax bits)
  unsigned long long* resid;  // [B][stride_ncr]: fixed-point sum of the draw weights
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
// Bounded wait for the phase with the given parity; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, unsigned bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void sts128(void* p, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
               ::"r"(smem_u32(p)), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
  return v;
}
// Atomic add with release semantics: publishes this thread's earlier writes
// (the partials of the items it counts).  The last arriver then issues
// fence_acquire() before reading the other arrivers' partials; the other
// arrivers need no acquire, and later memory operations do not wait for the
// atomic.
__device__ __forceinline__ unsigned int atom_add_release(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_acquire() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ unsigned int ld_relaxed(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
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
__device__ __forceinline__ uint32_t vec_word(const uint4& v, int q) {
  return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}
// per-half equality of two bf16 pairs (0xffff in each equal half)
__device__ __forceinline__ uint32_t bf16x2_eq(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 128-bit atomics on global memory: a 16-byte exchange, and a 16-byte read as
// a compare-and-swap of zero with zero (it never changes the value).
__device__ __forceinline__ void atom_store_b128(void* p, uint4 v) {
  const unsigned long long lo = ((unsigned long long)v.y << 32) | v.x;
  const unsigned long long hi = ((unsigned long long)v.w << 32) | v.z;
  asm volatile(
      "{\n .reg .b128 nv, ov;\n mov.b128 nv, {%1, %2};\n"
      " atom.relaxed.gpu.global.exch.b128 ov, [%0], nv;\n}\n"
      ::"l"(p), "l"(lo), "l"(hi) : "memory");
}
__device__ __forceinline__ uint4 atom_load_b128(const void* p) {
  unsigned long long lo, hi;
  const unsigned long long z = 0ull;
  asm volatile(
      "{\n .reg .b128 cz, ov;\n mov.b128 cz, {%2, %2};\n"
      " atom.relaxed.gpu.global.cas.b128 ov, [%3], cz, cz;\n mov.b128 {%0, %1}, ov;\n}\n"
      : "=l"(lo), "=l"(hi) : "l"(z), "l"(p) : "memory");
  return make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
}

__device__ __forceinline__ void write_record(DecRecord* r, int b, const Decision& d) {
  const uint32_t tag = kDecTag | ((uint32_t)d.reject << 8) | (uint32_t)d.k;
  atom_store_b128(&r->tag_b, make_uint4(tag, __float_as_uint(d.inv_st), __float_as_uint(d.rho), 0u));
  atom_store_b128(&r->tag_a, make_uint4(tag, (uint32_t)b, __float_as_uint(d.mt), __float_as_uint(d.md)));
}

// A published record (both halves, one round trip): its request and decision
// (without the temperature constants).  False while it is not yet complete.
__device__ __forceinline__ bool read_record(const DecRecord* r, int& b, Decision& d) {
  const uint4 a = atom_load_b128(&r->tag_a);
  const uint4 h = atom_load_b128(&r->tag_b);
  if (!(a.x & kDecTag) || a.x != h.x) return false;
  d.k = (int)(a.x & 0xffu);
  d.reject = (int)((a.x >> 8) & 1u);
  b = (int)a.y;
  d.mt = __uint_as_float(a.z);
  d.md = __uint_as_float(a.w);
  d.inv_st = __uint_as_float(h.y);
  d.rho = __uint_as_float(h.z);
  return true;
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

// (A temperature of exactly 0 selects the greedy steps and never gets here.)
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

__device__ __forceinline__ int clamp_gamma(int g, int G) { return g < 0 ? 0 : (g > G ? G : g); }

// Where request b's data lives.  Padded layout: target rows b (G+1) + i,
// draft rows, tokens and p/q entries b G + i, uniforms b (G+1) + i with the
// final draw's in column G.  Packed layout (cu = prefix of the draft
// lengths): draft rows, tokens and p/q entries cu[b] + i, target rows and
// uniforms cu[b] + b + i with the final draw's at i = gamma_b.  A packed
// request whose prefix is inconsistent (cu[b] < 0, cu[b+1] < cu[b],
// cu[b+1] > total or a length above G) is flagged and given no drafts, with
// its offset clamped into the arrays, so no access leaves them.
struct ReqAddr {
  size_t t0;   // first target row
  size_t d0;   // first draft row, token and p/q entry
  size_t u0;   // first acceptance uniform
  size_t uf;   // the final draw's uniform
  int gb;      // draft length
  unsigned int flags;
};
__device__ __forceinline__ int packed_base(const Params& P, int b, int& gb, unsigned int& flags) {
  const int c0 = P.cu[b], c1 = P.cu[b + 1];
  const bool ok = 0 <= c0 && c0 <= c1 && c1 <= P.total && c1 - c0 <= P.G;
  if (!ok) flags |= SV_STATUS_BAD_GAMMA;
  gb = ok ? c1 - c0 : 0;
  return ok ? c0 : (c0 < 0 ? 0 : (c0 > P.total ? P.total : c0));
}
template <bool PK>
__device__ __forceinline__ ReqAddr addr_from_base(const Params& P, int b, int base, int gb) {
  ReqAddr a;
  a.flags = 0;
  a.gb = gb;
  if constexpr (PK) {
    a.d0 = (size_t)base;
    a.t0 = (size_t)base + (size_t)(P.b_base + b);
    a.u0 = a.t0;
    a.uf = a.t0 + (size_t)gb;
  } else {
    a.d0 = (size_t)b * (size_t)P.G;
    a.t0 = (size_t)b * (size_t)(P.G + 1);
    a.u0 = a.t0;
    a.uf = a.t0 + (size_t)P.G;
  }
  return a;
}
template <bool PK>
__device__ __forceinline__ ReqAddr req_addr(const Params& P, int b) {
  unsigned int flags = 0;
  int gb = 0, base = 0;
  if constexpr (PK) {
    base = packed_base(P, b, gb, flags);
  } else {
    const int g_in = P.gamma ? P.gamma[b] : 0;
    gb = clamp_gamma(g_in, P.G);
    if (g_in != gb) flags |= SV_STATUS_BAD_GAMMA;
  }
  ReqAddr a = addr_from_base<PK>(P, b, base, gb);
  a.flags = flags;
  return a;
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
// Draw weights (shared by R items and the final in-chunk scan)
// After a rejection at k the weight of a token is the residual
// r = max(0, p - q) = (1/S_t) * max(0, e_t - e_d * S_t/S_d); for the bonus
// draw it is p = e_t / S_t.  Weights are kept in 2^39 fixed point so that
// chunk sums are exact and independent of summation order.
// ---------------------------------------------------------------------------
struct ResidC {
  float mt, md, inv_st, rho, hi, lo;
  int reject;
  float c16;   // inv_st * 2^23 (exact): a weight in units of 2^-23
  float nrho;  // -rho
};
__device__ __forceinline__ void resid_scales(ResidC& k) {
  k.c16 = __fmul_rn(k.inv_st, 8388608.0f);
  k.nrho = -k.rho;
}

// A weight w in [0, 1] is used in 2^39 fixed point, round(w 2^39), computed
// from y = w 2^23 with float and 32-bit integer operations only (the
// float-to-integer conversions run at a fraction of the ALU rate on this
// GPU).  Adding 2^23 rounds y to an integer held in the low mantissa bits,
// t = RN(y + 2^23); the remainder y - (t - 2^23) is exact, and 2^16 times it
// is rounded the same way with 1.5 * 2^23 (which also covers negative
// values): t2 = RN(2^16 (y - (t - 2^23)) + 1.5 * 2^23).  Then
// round(w 2^39) = 2^16 (bits(t) - bits(2^23)) + (bits(t2) - bits(1.5 * 2^23)),
// ties to even in both steps.  Valid for 0 <= y <= 2^23 (a little more is
// fine).
struct FixParts {
  float t, t2;
};
__device__ __forceinline__ FixParts fix_parts(float y) {
  const float t = __fadd_rn(y, 8388608.0f);
  const float dl = __fsub_rn(y, __fadd_rn(t, -8388608.0f));
  return FixParts{t, __fmaf_rn(dl, 65536.0f, 12582912.0f)};
}
__device__ __forceinline__ unsigned long long fix_round(float y) {
  const FixParts f = fix_parts(y);
  const uint32_t yr = __float_as_uint(f.t) - 0x4b000000u;
  const int rr = (int)(__float_as_uint(f.t2) - 0x4b400000u);
  return ((unsigned long long)yr << 16) + (unsigned long long)(long long)rr;
}

// Sums of round(w 2^39) over many weights, as two 32-bit sums of raw float
// bits (of t and t2 above); the constant offsets are removed once per sum.
// Exact while the true sum stays below 2^48 (here at most 64 terms of
// <= 2^39 per sum).
struct FixAcc {
  uint32_t hi, lo, n;
};
__device__ __forceinline__ void fix_add_parts(FixAcc& a, float t, float t2) {
  a.hi += __float_as_uint(t);
  a.lo += __float_as_uint(t2);
  ++a.n;
}
__device__ __forceinline__ void fix_add(FixAcc& a, float y) {
  const FixParts f = fix_parts(y);
  fix_add_parts(a, f.t, f.t2);
}
__device__ __forceinline__ unsigned long long fix_value(const FixAcc& a) {
  const uint32_t hs = a.hi - a.n * 0x4b000000u;
  const int ls = (int)(a.lo - a.n * 0x4b400000u);
  return ((unsigned long long)hs << 16) + (unsigned long long)(long long)ls;
}

// The draw weight of one token, y = w 2^23, before rounding.  The packed
// residual path performs the same operations pair by pair.
template <bool REJECT>
__device__ __forceinline__ float draw_x(float zt, float zd, const ResidC& k) {
  const float et = ex2_approx(exp_arg(zt, k.mt, k.hi, k.lo));
  float v = et;
  if (REJECT) {
    const float ed = ex2_approx(exp_arg(zd, k.md, k.hi, k.lo));
    v = fmaxf(__fmaf_rn(ed, k.nrho, et), 0.0f);
  }
  return __fmul_rn(v, k.c16);
}

template <bool REJECT>
__device__ __forceinline__ unsigned long long draw_weight(float zt, float zd, const ResidC& k) {
  return fix_round(draw_x<REJECT>(zt, zd, k));
}

__device__ __forceinline__ unsigned long long draw_weight(float zt, float zd, const ResidC& k) {
  return k.reject ? draw_weight<true>(zt, zd, k) : draw_weight<false>(zt, zd, k);
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
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
// (a.hi + a.lo) * (bh + bl)
__device__ __forceinline__ FF ff_mul(FF a, float bh, float bl) {
  const float p = __fmul_rn(a.hi, bh);
  const float e = __fmaf_rn(a.hi, bh, -p);
  const float t = __fmaf_rn(a.hi, bl, __fmaf_rn(a.lo, bh, e));
  return ff_fast_two_sum(p, t);
}
// (a.hi + a.lo) / (b.hi + b.lo), rounded to float (within about one ulp)
__device__ __forceinline__ float ff_div(FF a, FF b) {
  const float q = __fdiv_rn(a.hi, b.hi);
  const float r = __fmaf_rn(-q, b.hi, a.hi);  // exact remainder of the leading quotient
  const float c = __fmaf_rn(-q, b.lo, __fadd_rn(r, a.lo));
  return __fadd_rn(q, __fdiv_rn(c, b.hi));
}

// Shuffle of a float-float value.
__device__ __forceinline__ FF shfl_xor_ff(FF v, int o) {
  return FF{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}

// Where a request's per-item partials are read from: slot s (target row s, or
// draft row i at slot G + 1 + i), item c.
struct GlobalParts {  // the workspace: written by other SMs, so read past L1
  const float2* p;
  size_t stride;
  __device__ __forceinline__ float2 operator()(int slot, int c) const {
    return __ldcg(p + (size_t)slot * stride + (size_t)c);
  }
};
struct SharedParts {  // this CTA's shared memory
  const float2* p;
  int stride;
  __device__ __forceinline__ float2 operator()(int slot, int c) const {
    return p[slot * stride + c];
  }
};
struct RowParts {  // a copy of one row's partials (the slot is implied)
  const float2* p;
  __device__ __forceinline__ float2 operator()(int, int c) const { return p[c]; }
};
__device__ __forceinline__ GlobalParts global_parts(const Params& P, int b) {
  return GlobalParts{P.stats + (size_t)b * (2 * P.G + 1) * P.stride_nc, (size_t)P.stride_nc};
}

// The per-item partials of a request's rows are reduced eight rows at a time:
// lanes 4r..4r+3 take row r of the group, each every fourth chunk (up to
// kHeld chunks held in registers, the rest in a tail loop).  The code is kept
// compact: it runs once per request, usually with a cold instruction cache.
constexpr int kHeld = 10;

// Row statistics (sampling): M = max, S = sum_c s_c 2^((m_c - M) c) in
// float-float, written to rs[x] (M), rs[64 + x] (S hi), rs[128 + x] (S lo),
// x = i for target row i and gamma_b + 1 + i for draft row i.  The rows are
// those of positions [lo, hi) (target, then draft) and, if `bonus`, target
// row gamma_b; a row's arithmetic does not depend on which others share the
// call.
template <int EB, class Parts>
__device__ __forceinline__ unsigned int row_stats(const Params& P, const Parts& parts, int gb,
                                                  TempC tc, float* rs, int lo, int hi,
                                                  bool bonus) {
  const int G = P.G, NC = P.NC;
  const int lane = threadIdx.x & 31, part = lane & 3;
  const int npos = hi - lo;
  const int nrows = 2 * npos + (bonus ? 1 : 0);
  const float2 none = make_float2(-INFINITY, 0.0f);
  unsigned int flags = 0;
#pragma unroll 1
  for (int r0 = 0; r0 < nrows; r0 += 8) {
    const int r = r0 + (lane >> 2);
    const bool live = r < nrows;
    // the row: target lo + r, draft lo + r - npos, or the bonus row
    const int ti = r < npos ? lo + r : (r < 2 * npos ? -1 : gb);
    const int di = lo + r - npos;
    const int slot = !live ? 0 : (ti >= 0 ? ti : G + 1 + di);
    const int x = ti >= 0 ? ti : gb + 1 + di;
    float2 v[kHeld];
#pragma unroll
    for (int j = 0; j < kHeld; ++j) {
      const int c = part + 4 * j;
      v[j] = (live && c < NC) ? parts(slot, c) : none;
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kHeld; ++j) m = fmaxf(m, v[j].x);
#pragma unroll 1
    for (int c = part + 4 * kHeld; live && c < NC; c += 4) m = fmaxf(m, parts(slot, c).x);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    FF S{0.0f, 0.0f};
    if (m > -INFINITY) {
#pragma unroll
      for (int j = 0; j < kHeld; ++j)
        if (v[j].x > -INFINITY)
          S = ff_add(S, FF{__fmul_rn(v[j].y, ex2_approx(exp_arg(v[j].x, m, tc.hi, tc.lo))), 0.0f});
#pragma unroll 1
      for (int c = part + 4 * kHeld; live && c < NC; c += 4) {
        const float2 ms = parts(slot, c);
        if (ms.x > -INFINITY)
          S = ff_add(S, FF{__fmul_rn(ms.y, ex2_approx(exp_arg(ms.x, m, tc.hi, tc.lo))), 0.0f});
      }
    }
    S = ff_add(S, shfl_xor_ff(S, 1));
    S = ff_add(S, shfl_xor_ff(S, 2));
    if (live && part == 0) {
      if (!isfinite(m) || !(S.hi > 0.0f)) flags |= SV_STATUS_NONFINITE_ROW;
      rs[x] = m;
      rs[64 + x] = S.hi;
      rs[128 + x] = S.lo;
    }
  }
  __syncwarp();
  return flags;
}

// ---------------------------------------------------------------------------
// Per-request decision (sampling), run by one warp: the one that completed
// the request's last A item.  Float and float-float arithmetic only on the
// common path; float64 appears where an exponent is extreme and for the
// optional probability outputs.  rs: 192 floats of the warp's free shared
// staging buffer.
// ---------------------------------------------------------------------------

// Float-float helpers for the bonus draw: warp inclusive scan and order.
__device__ __forceinline__ FF warp_incl_scan_ff(FF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    FF y;
    y.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
    y.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
    if (lane >= o) v = ff_add(v, y);
  }
  return v;
}
__device__ __forceinline__ bool ff_le(FF a, FF b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo <= b.lo);
}
__device__ __forceinline__ FF ff_sub(FF a, FF b) { return ff_add(a, FF{-b.hi, -b.lo}); }

// Bonus draw (every draft accepted): the token comes from p of target row gb,
// whose per-item partials (m_c, s_c) the A pass already wrote, so no R pass
// is needed.  Chunk weights W_c = s_c 2^((m_c - M) c) and their float-float
// prefix sums locate the A chunk holding u S (past the total, from rounding:
// the last chunk of positive weight).  Inside that chunk the weights are
// taken in exact 2^39 fixed point relative to W_c and the token is the
// smallest whose prefix exceeds floor(r F), r = (u S - prefix) / W_c and F
// the chunk's fixed-point total: lane sums, a warp scan and one 16-token
// vector, with no serial walk.  The CDF is accurate to about 1e-7 of S, like
// the residual path's.
template <int EB, bool PK, class Parts>
__device__ __noinline__ void final_bonus(const Params& P, const Parts& parts, int b, int gb,
                                         TempC tc, float M, unsigned char* stage) {
  constexpr int AE = kItemBytes / EB;  // logits per A chunk
  constexpr int EPL = AE / 32;         // contiguous logits per lane
  constexpr int VEC = 16 / EB;
  constexpr int NV = EPL / VEC;        // 16-byte vectors per lane
  const int G = P.G, V = P.V, NC = P.NC;
  const int lane = threadIdx.x & 31;
  unsigned int flags = 0;
  const ReqAddr A = req_addr<PK>(P, b);
  const float u = sanitize_uniform(P.uniforms[A.uf], flags);
  auto chunk_w = [&](int c) -> float {
    const float2 ms = parts(gb, c);
    return ms.x > -INFINITY ? __fmul_rn(ms.y, ex2_approx(exp_arg(ms.x, M, tc.hi, tc.lo))) : 0.0f;
  };
  // 1. the chunk: lane l owns chunks [c0, c1)
  const int cpl = (NC + 31) >> 5;
  const int c0 = min(NC, lane * cpl), c1 = min(NC, c0 + cpl);
  FF own{0.0f, 0.0f};
#pragma unroll 1
  for (int c = c0; c < c1; ++c) own = ff_add(own, FF{chunk_w(c), 0.0f});
  FF incl = warp_incl_scan_ff(own);
  FF tot;
  tot.hi = __shfl_sync(0xffffffffu, incl.hi, 31);
  tot.lo = __shfl_sync(0xffffffffu, incl.lo, 31);
  const FF target = ff_mul(tot, u, 0.0f);
  int cs = NC - 1;
  FF base{0.0f, 0.0f};
  {
    const FF excl = ff_sub(incl, own);
    const unsigned int hit = __ballot_sync(0xffffffffu, c0 < c1 && ff_le(excl, target) &&
                                                        !ff_le(incl, target));
    int l = hit ? __ffs(hit) - 1 : -1;
    int csl = -1;
    FF run = excl;
    if (lane == l) {
#pragma unroll 1
      for (int c = c0; c < c1; ++c) {
        const FF nxt = ff_add(run, FF{chunk_w(c), 0.0f});
        if (!ff_le(nxt, target)) {
          csl = c;
          break;
        }
        run = nxt;
      }
    }
    if (l >= 0) {
      cs = __shfl_sync(0xffffffffu, csl, l);
      base.hi = __shfl_sync(0xffffffffu, run.hi, l);
      base.lo = __shfl_sync(0xffffffffu, run.lo, l);
    }
    if (l < 0 || cs < 0) {
      // u S at or past the total (rounding): the last chunk of positive
      // weight, from its start (the walk below then takes its last token of
      // positive weight)
      int lastc = -1;
      FF before{0.0f, 0.0f}, r2 = excl;
#pragma unroll 1
      for (int c = c0; c < c1; ++c) {
        const float w = chunk_w(c);
        if (w > 0.0f) {
          lastc = c;
          before = r2;
        }
        r2 = ff_add(r2, FF{w, 0.0f});
      }
      const unsigned int has = __ballot_sync(0xffffffffu, lastc >= 0);
      if (has) {
        const int hl = 31 - __clz(has);
        cs = __shfl_sync(0xffffffffu, lastc, hl);
        base.hi = __shfl_sync(0xffffffffu, before.hi, hl);
        base.lo = __shfl_sync(0xffffffffu, before.lo, hl);
      } else {
        cs = NC - 1;  // no weight at all (flagged as a non-finite row)
        base = FF{0.0f, 0.0f};
      }
    }
  }

  // 2. the token inside chunk cs, exactly: its weights in 2^39 fixed point
  //    relative to the chunk's weight W (y = w 2^23 / W), and the position
  //    r = (u S - base) / W of u S inside the chunk as a float in [0, 1); the
  //    token is the smallest one whose fixed-point prefix exceeds floor(r F),
  //    F the chunk's fixed-point total.  Lane l owns the chunk's logits
  //    [l EPL, (l + 1) EPL), staged through shared memory (vectors swizzled per
  //    lane; scalar loads where the row does not allow 16-byte vectors, -inf past
  //    its end).
  const char* row = P.target + (A.t0 + (size_t)gb) * (size_t)V * EB;
  auto slot_of = [&](int q) { return (lane * NV + (q ^ (lane & (NV - 1)))) * 16; };
  const size_t e0 = (size_t)cs * AE + (size_t)lane * EPL;
  {
    const bool vec_ok = (reinterpret_cast<uintptr_t>(row) & 15) == 0 && e0 + EPL <= (size_t)V;
    if (vec_ok) {
#pragma unroll 4
      for (int q = 0; q < NV; ++q)
        sts128(stage + slot_of(q), __ldcg(reinterpret_cast<const uint4*>(row + (e0 + (size_t)q * VEC) * EB)));
    } else {
#pragma unroll 1
      for (int q = 0; q < NV; ++q) {
        uint32_t w[4];
#pragma unroll 1
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
        sts128(stage + slot_of(q), make_uint4(w[0], w[1], w[2], w[3]));
      }
    }
  }
  const float W = chunk_w(cs);
  ResidC kc;  // the bonus weight, scaled to the chunk: y = 2^((z - M) c) 2^23 / W
  kc.mt = M;
  kc.md = 0.0f;
  kc.inv_st = W > 0.0f ? __fdiv_rn(1.0f, W) : 0.0f;
  kc.rho = 0.0f;
  resid_scales(kc);
  kc.hi = tc.hi;
  kc.lo = tc.lo;
  kc.reject = 0;
  float r = W > 0.0f ? ff_div(ff_sub(target, base), FF{W, 0.0f}) : 0.0f;
  r = fminf(fmaxf(r, 0.0f), 0.99999994f);  // the largest float below 1
  auto vec_sum = [&](int q) -> unsigned long long {
    const uint4 t = lds128(stage + slot_of(q));
    FixAcc a{0u, 0u, 0u};
#pragma unroll
    for (int h = 0; h < VEC; ++h) fix_add(a, draw_x<false>(vec_elem<EB>(t, h), -INFINITY, kc));
    return fix_value(a);
  };
  unsigned long long lsum = 0;
#pragma unroll 1
  for (int q = 0; q < NV; ++q) lsum += vec_sum(q);
  const unsigned long long li = warp_incl_scan_u64(lsum);
  const unsigned long long Ftot = __shfl_sync(0xffffffffu, li, 31);
  const unsigned long long t = scaled_target(r, Ftot);  // < Ftot when Ftot > 0
  int tok = -1;
  unsigned long long run = li - lsum;
  if (Ftot > 0ull && run <= t && t < li) {
#pragma unroll 1
    for (int q = 0; q < NV && tok < 0; ++q) {
      const unsigned long long vs = vec_sum(q);
      if (run + vs > t) {
        const uint4 tv = lds128(stage + slot_of(q));
#pragma unroll
        for (int h = 0; h < VEC; ++h) {
          const unsigned long long wv = draw_weight<false>(vec_elem<EB>(tv, h), -INFINITY, kc);
          if (tok < 0 && run + wv > t) tok = (int)(e0 + (size_t)(q * VEC + h));
          run += wv;
        }
      } else {
        run += vs;
      }
    }
  }
  const unsigned int holder = __ballot_sync(0xffffffffu, tok >= 0);
  tok = holder ? __shfl_sync(0xffffffffu, tok, __ffs(holder) - 1) : -1;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (lane == 0) {
    if (tok < 0) {
      flags |= SV_STATUS_INTERNAL;
      tok = V - 1;
    }
    P.out_tokens[(size_t)b * (G + 1) + gb] = tok;
    if (flags) atomicOr(P.status, flags);
  }
  __syncwarp();
}

// 2^e / S in float64, e and S float-float (the probability p(x) or q(x)).
__device__ __noinline__ double prob_f64(FF e, FF S) {
  if (!(e.hi > -INFINITY)) return 0.0;
  const float n = rintf(e.hi);
  const float f = __fadd_rn(__fsub_rn(e.hi, n), e.lo);
  const float v = __fmul_rn(ex2_approx(f), ff_div(FF{1.0f, 0.0f}, S));
  return ldexp((double)v, (int)fmaxf(n, -2000.0f));
}

// q(x) = 2^e / S is 0 in float64 (only reachable for e far below -1000).
__device__ __noinline__ bool q_underflows(FF e, FF S) {
  return exp2((double)e.hi + (double)e.lo) / ((double)S.hi + (double)S.lo) == 0.0;
}

// Request b's drafted tokens, their acceptance uniforms and the target and
// draft logits at them: lane i < gamma_b holds position i.
struct DraftIn {
  int x;
  float u, zt, zd;
  unsigned int flags;
};
template <int EB>
__device__ __forceinline__ DraftIn gather_drafts(const Params& P, const ReqAddr& A, int gb) {
  const int i = threadIdx.x & 31, V = P.V;
  DraftIn g{0, 0.0f, 0.0f, 0.0f, 0u};
  if (i < gb) {
    g.x = P.tokens[A.d0 + i];
    g.u = sanitize_uniform(P.uniforms[A.u0 + i], g.flags);
    if (g.x < 0 || g.x >= V) {
      g.flags |= SV_STATUS_BAD_TOKEN;
      g.x = g.x < 0 ? 0 : V - 1;
    }
    g.zt = load_elem<EB>(P.target, (A.t0 + i) * (size_t)V + (size_t)g.x);
    g.zd = load_elem<EB>(P.draft, (A.d0 + i) * (size_t)V + (size_t)g.x);
  }
  return g;
}

// The acceptance tests of request b at positions [lo, hi) from the row
// statistics of those positions (and of the bonus row gamma_b, if `bonus`),
// every earlier position having been accepted.  Returns k, the first
// rejected position (gamma_b when every draft is accepted and the bonus row
// is in), on every lane with the decision on lane 0; or -1 when all of
// [lo, hi) are accepted and later positions remain to be tested.  When emit
// is set it writes p/q of [lo, hi) and, once k is known, out_tokens (all but
// position k), num_accepted, p/q NaN past hi, and status.  One call over
// [0, gamma_b) with the bonus row is the whole decision.
template <int EB, bool PK, class Parts>
__device__ __forceinline__ int decide_range(const Params& P, const Parts& parts, int b, int gb,
                                            TempC tc, float* rs, const ReqAddr& A,
                                            const DraftIn& g, Decision& d, int lo, int hi,
                                            bool bonus, bool emit) {
  const int G = P.G;
  const int lane = threadIdx.x & 31;
  const int i = lane;
  const int x = g.x;
  const float u = g.u, zt = g.zt, zd = g.zd;
  unsigned int flags = lo == 0 ? g.flags : 0u;
  flags |= row_stats<EB>(P, parts, gb, tc, rs, lo, hi, bonus);

  // Acceptance test per position (lane i), then the first-reject ballot.
  // ratio p/q = 2^(e_t - e_d) * S_d / S_t with e = (z - m) log2(e)/T in
  // float-float; 2^(e_t - e_d) = 2^n * 2^f with |f| <= 1/2.
  bool reject = false;
  double p = NAN, q = NAN;
  if (i >= lo && i < hi) {
    const float mt = rs[i], md = rs[gb + 1 + i];
    const FF st{rs[64 + i], rs[128 + i]}, sd{rs[64 + gb + 1 + i], rs[128 + gb + 1 + i]};
    const FF et = ff_mul(ff_two_sum(zt, -mt), tc.hi, tc.lo);  // log2 of S_t p(x)
    const FF ed = ff_mul(ff_two_sum(zd, -md), tc.hi, tc.lo);  // log2 of S_d q(x)
    bool accept;
    if (!(zd > -INFINITY)) {
      accept = true;  // q(x) = 0 accepts
    } else if (!(zt > -INFINITY)) {
      accept = false;  // p(x) = 0: the ratio is 0
    } else if (ed.hi < -1000.0f && q_underflows(ed, sd)) {
      accept = true;  // q(x) is 0 in float64
    } else {
      const FF e = ff_add(et, FF{-ed.hi, -ed.lo});
      float ratio;
      if (e.hi >= 256.0f) {
        ratio = INFINITY;
      } else if (e.hi <= -256.0f) {
        ratio = 0.0f;
      } else {
        const float n = rintf(e.hi);
        const float f = __fadd_rn(__fsub_rn(e.hi, n), e.lo);
        ratio = ldexpf(__fmul_rn(ex2_approx(f), ff_div(sd, st)), (int)n);
      }
      accept = u < ratio;
    }
    reject = !accept;
    if (emit && (P.p_tok || P.q_tok)) {
      p = (zt > -INFINITY) ? prob_f64(et, st) : 0.0;
      q = (zd > -INFINITY) ? prob_f64(ed, sd) : 0.0;
    }
  }
  const unsigned int rej = __ballot_sync(0xffffffffu, reject);
  const int k = rej ? (__ffs(rej) - 1) : (bonus ? gb : -1);
  if (emit && k >= 0 && i <= G && i != k) P.out_tokens[(size_t)b * (G + 1) + i] = i < k ? x : -1;
  // packed p/q hold this request's gb entries only
  if (emit && i >= lo && i < (PK ? gb : G) && (k >= 0 || i < hi)) {
    const bool evaluated = i < hi && (k < 0 || i <= k);
    if (P.p_tok) P.p_tok[A.d0 + i] = evaluated ? p : NAN;
    if (P.q_tok) P.q_tok[A.d0 + i] = evaluated ? q : NAN;
  }
  const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
  if (emit && lane == 0 && any) atomicOr(P.status, any);
  if (k < 0) return k;
  if (lane == 0) {
    const int kd = gb + 1 + (k < gb ? k : 0);
    const FF st_k{rs[64 + k], rs[128 + k]}, sd_k{rs[64 + kd], rs[128 + kd]};
    if (emit && P.num_accepted) P.num_accepted[b] = k;
    d.k = k;
    d.reject = k < gb ? 1 : 0;
    d.mt = rs[k];
    d.md = d.reject ? rs[kd] : 0.0f;
    d.inv_st = ff_div(FF{1.0f, 0.0f}, st_k);
    d.rho = d.reject ? ff_div(st_k, sd_k) : 0.0f;
    d.c_hi = tc.hi;
    d.c_lo = tc.lo;
  }
  return k;
}

template <int EB, bool PK, class Parts>
__device__ __forceinline__ int decide_core(const Params& P, const Parts& parts, int b, int gb,
                                           TempC tc, float* rs, const ReqAddr& A,
                                           const DraftIn& g, Decision& d, bool emit = true) {
  return decide_range<EB, PK>(P, parts, b, gb, tc, rs, A, g, d, 0, gb, true, emit);
}

// Sampling decision on the persistent path, run by the warp that completed
// request b's last A item: publishes a reject to the decision record and the
// queue, or draws the bonus token itself.
template <int EB, bool PK>
__device__ __noinline__ void decide_sample(const Params& P, int b, int gb, TempC tc, float* rs) {
  const int lane = threadIdx.x & 31;
  const ReqAddr A = req_addr<PK>(P, b);
  // the drafted tokens, their uniforms and logits are requested first
  const DraftIn g = gather_drafts<EB>(P, A, gb);
  Decision d;
  const GlobalParts parts = global_parts(P, b);
  const int k = decide_core<EB, PK>(P, parts, b, gb, tc, rs, A, g, d);
  if (lane == 0) {
    P.cnt_a[b] = 0;
    if (d.reject) {
      // R work: the decision goes to the request's record and the queue
      write_record(&P.dec[b], b, d);
      write_record(&P.queue[atomicAdd(P.q_tail, 1u)], b, d);
    }
  }
  __syncwarp();
  if (k == gb) final_bonus<EB, PK>(P, parts, b, gb, tc, rs[gb], reinterpret_cast<unsigned char*>(rs));
  if (lane == 0) {
    __threadfence();  // a queue entry is visible before the count that covers it
    atomicAdd(P.dec_count, 1u);
  }
  __syncwarp();
}

// Greedy decision: argmax per target row from the per-item partials (rows
// reduced eight at a time as above; rs holds the row argmaxes), then the
// first mismatch by warp ballot.
// Greedy steps over target rows [lo, hi) (hi <= gamma_b + 1), every earlier
// draft having matched its row's argmax: rs[r] receives row r's argmax.
// Returns k, the first position in [lo, hi) whose draft differs from the
// argmax (gamma_b when every draft matches and row gamma_b is in), or -1 when
// all of [lo, hi) match and later rows remain.  Once k is known it writes
// out_tokens (the drafts before k, the argmax at k, then -1), num_accepted,
// NaN p/q and status.  One call over [0, gamma_b + 1) is the whole step.
template <bool PK, class Parts>
__device__ __forceinline__ int greedy_range(const Params& P, const Parts& parts, int b, int gb,
                                            int* rs, int lo, int hi) {
  const int G = P.G, V = P.V, NC = P.NC;
  const int lane = threadIdx.x & 31, part = lane & 3;
  unsigned int flags = 0;
  const int i = lane;
  const ReqAddr A = req_addr<PK>(P, b);
  int x = 0;
  if (i < gb) x = P.tokens[A.d0 + i];
#pragma unroll 1
  for (int r0 = lo; r0 < hi; r0 += 8) {
    const int r = r0 + (lane >> 2);
    const bool live = r < hi;
    const int slot = live ? r : 0;
    float2 v[kHeld];
#pragma unroll
    for (int j = 0; j < kHeld; ++j) {
      const int c = part + 4 * j;
      v[j] = (live && c < NC) ? parts(slot, c) : make_float2(-INFINITY, __int_as_float(0x7fffffff));
    }
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kHeld; ++j) argmax_combine(bv, bi, v[j].x, __float_as_int(v[j].y));
#pragma unroll 1
    for (int c = part + 4 * kHeld; live && c < NC; c += 4) {
      const float2 mi = parts(slot, c);
      argmax_combine(bv, bi, mi.x, __float_as_int(mi.y));
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_combine(bv, bi, v2, i2);
    }
    if (live && part == 0) {
      if (!isfinite(bv)) flags |= SV_STATUS_NONFINITE_ROW;
      rs[r] = (bi >= 0 && bi < V) ? bi : 0;
    }
  }
  __syncwarp();
  bool mismatch = false;
  if (lo == 0 && i < gb && (x < 0 || x >= V)) flags |= SV_STATUS_BAD_TOKEN;
  if (i >= lo && i < hi && i < gb) mismatch = x != rs[i];
  const unsigned int mm = __ballot_sync(0xffffffffu, mismatch);
  const int k = mm ? (__ffs(mm) - 1) : (hi > gb ? gb : -1);
  const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && any) atomicOr(P.status, any);
  if (k < 0) return k;
  const int gk = rs[k];
  if (i <= G) P.out_tokens[(size_t)b * (G + 1) + i] = i < k ? x : (i == k ? gk : -1);
  if (i < (PK ? gb : G)) {  // a sampling call's zero-temperature request has no p or q
    if (P.p_tok) P.p_tok[A.d0 + i] = NAN;
    if (P.q_tok) P.q_tok[A.d0 + i] = NAN;
  }
  if (lane == 0 && P.num_accepted) P.num_accepted[b] = k;
  __syncwarp();
  return k;
}
template <bool PK, class Parts>
__device__ __forceinline__ void greedy_core(const Params& P, const Parts& parts, int b, int gb,
                                            int* rs) {
  (void)greedy_range<PK>(P, parts, b, gb, rs, 0, gb + 1);
}
template <bool PK>
__device__ __noinline__ void decide_greedy(const Params& P, int b, int gb, int* rs) {
  greedy_core<PK>(P, global_parts(P, b), b, gb, rs);
  if ((threadIdx.x & 31) == 0) P.cnt_a[b] = 0;
  __syncwarp();
}

// Sum over R chunk c of the draw weights, read from global memory by the
// whole warp.
template <int EB>
__device__ unsigned long long chunk_weight_sum(const char* trow, const char* drow, int V, int c,
                                               const ResidC& kc) {
  constexpr int RE = kHalfBytes / EB;
  const int lane = threadIdx.x & 31;
  unsigned long long s = 0;
  const int e1 = min(V, (c + 1) * RE);
  for (int e = c * RE + lane; e < e1; e += 32)
    s += draw_weight(load_elem<EB>(trow, (size_t)e), drow ? load_elem<EB>(drow, (size_t)e) : -INFINITY, kc);
  return warp_sum_u64(s);
}

// The final draw from R chunk sums rp[0..NCR) of target row trow (and, after a
// reject, draft row drow), run by one warp: the chunk whose prefix passes
// floor(u S), then a scan of that chunk only, staged in `stage` (8 KB).  When
// the sums vanish in fixed point (p_k and q_k agree within its resolution)
// the draw uses p_k: its chunk sums replace the residual ones in rp.  GSUMS:
// rp is in global memory, written by other SMs (read past L1); otherwise in
// this CTA's shared memory.  Returns the token, or -1 (an internal error).
template <int EB, bool GSUMS>
__device__ __forceinline__ int chunk_draw(const char* trow, const char* drow, int V, int NCR,
                                          float u_s, ResidC kc, unsigned long long* rp,
                                          unsigned char* stage) {
  constexpr int RE = kHalfBytes / EB;  // elements per R chunk
  constexpr int EPL = RE / 32;         // contiguous elements per lane in the scan
  constexpr int VEC = 16 / EB;
  constexpr int NV = EPL / VEC;        // vectors per lane per row (8)
  const int lane = threadIdx.x & 31;
  auto ld_sum = [&](int c) -> unsigned long long {
    if constexpr (GSUMS) return __ldcg(&rp[c]);
    else return rp[c];
  };

  // 1. The chunk: lane l owns chunks [c0, c1); a scan over the lanes' sums
  //    finds the lane, that lane walks its chunks.
  const int cpl = (NCR + 31) >> 5;
  const int c0 = min(NCR, lane * cpl), c1 = min(NCR, c0 + cpl);
  unsigned long long own = 0;
#pragma unroll 1
  for (int c = c0; c < c1; ++c) own += ld_sum(c);
  unsigned long long incl = warp_incl_scan_u64(own);
  unsigned long long S = __shfl_sync(0xffffffffu, incl, 31);
  if (S == 0ull) {
    // The residual vanished in fixed point (p_k and q_k agree within its
    // resolution): draw from p_k instead; its chunk sums replace the
    // residual ones.
    kc.reject = 0;
    drow = nullptr;
    own = 0;
#pragma unroll 1
    for (int c = 0; c < NCR; ++c) {
      const unsigned long long sc = chunk_weight_sum<EB>(trow, nullptr, V, c, kc);
      if (c >= c0 && c < c1) {
        rp[c] = sc;
        own += sc;
      }
    }
    incl = warp_incl_scan_u64(own);
    S = __shfl_sync(0xffffffffu, incl, 31);
  }
  const unsigned long long target = scaled_target(u_s, S);  // < S
  int cs = -1;
  unsigned long long base = 0;
  {
    const unsigned long long excl = incl - own;
    const unsigned int hit = __ballot_sync(0xffffffffu, excl <= target && target < incl);
    if (hit) {
      const int l = __ffs(hit) - 1;
      if (lane == l) {
        unsigned long long run = excl;
#pragma unroll 1
        for (int c = c0; c < c1; ++c) {
          const unsigned long long w = ld_sum(c);
          if (run + w > target) {
            cs = c;
            break;
          }
          run += w;
        }
        base = run;
      }
      cs = __shfl_sync(0xffffffffu, cs, l);
      base = __shfl_sync(0xffffffffu, base, l);
    }
  }

  // 2. The token inside chunk cs.  Every lane loads its EPL contiguous logits
  //    at once (scalar loads where the rows do not allow 16-byte vectors; -inf
  //    past the end of the row) into the warp's free staging buffer (target
  //    half, then draft half, vectors swizzled per lane), sums their weights,
  //    and the lane whose range holds the target walks to the token.
  int tok = -1;
  if (cs >= 0) {
    const size_t e0 = (size_t)cs * RE + (size_t)lane * EPL;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(trow) |
                          reinterpret_cast<uintptr_t>(drow)) & 15) == 0 &&
                        e0 + EPL <= (size_t)V;
    auto slot_of = [&](int q) { return (lane * NV + (q ^ (lane & (NV - 1)))) * 16; };
    if (vec_ok) {
      uint4 tv[NV], dv[NV];
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        tv[q] = __ldcg(reinterpret_cast<const uint4*>(trow + (e0 + (size_t)q * VEC) * EB));
        dv[q] = drow ? __ldcg(reinterpret_cast<const uint4*>(drow + (e0 + (size_t)q * VEC) * EB))
                     : neg_inf_vec(EB);
      }
#pragma unroll
      for (int q = 0; q < NV; ++q) {
        sts128(stage + slot_of(q), tv[q]);
        sts128(stage + kHalfBytes + slot_of(q), dv[q]);
      }
    } else {
      // element by element, -inf past the end of the row
#pragma unroll 1
      for (int q = 0; q < NV; ++q) {
        uint32_t w[2][4];
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const char* row = r ? drow : trow;
            if (EB == 2) {
              const size_t ea = e0 + (size_t)q * 8 + 2 * h, eb = ea + 1;
              const uint32_t lo = row && ea < (size_t)V ? reinterpret_cast<const unsigned short*>(row)[ea] : 0xff80u;
              const uint32_t hi = row && eb < (size_t)V ? reinterpret_cast<const unsigned short*>(row)[eb] : 0xff80u;
              w[r][h] = lo | (hi << 16);
            } else {
              const size_t e = e0 + (size_t)q * 4 + h;
              w[r][h] = row && e < (size_t)V ? __float_as_uint(reinterpret_cast<const float*>(row)[e])
                                              : 0xff800000u;
            }
          }
        }
        sts128(stage + slot_of(q), make_uint4(w[0][0], w[0][1], w[0][2], w[0][3]));
        sts128(stage + kHalfBytes + slot_of(q), make_uint4(w[1][0], w[1][1], w[1][2], w[1][3]));
      }
    }
    // A bonus draw runs the residual formula with a -inf draft row: the draft
    // term is exactly 0 and the weight equals the bonus weight bit for bit.
    FixAcc acc{0u, 0u, 0u};
#pragma unroll 1
    for (int q = 0; q < NV; ++q) {
      const uint4 t = lds128(stage + slot_of(q)), dd = lds128(stage + kHalfBytes + slot_of(q));
#pragma unroll
      for (int h = 0; h < VEC; ++h) fix_add(acc, draw_x<true>(vec_elem<EB>(t, h), vec_elem<EB>(dd, h), kc));
    }
    own = fix_value(acc);
    incl = warp_incl_scan_u64(own);
    unsigned long long run = base + incl - own;
    if (run <= target && target < run + own) {
      // this lane holds the token
#pragma unroll 1
      for (int q = 0; q < NV && tok < 0; ++q) {
        const uint4 t = lds128(stage + slot_of(q)), dd = lds128(stage + kHalfBytes + slot_of(q));
#pragma unroll
        for (int h = 0; h < VEC; ++h) {
          const unsigned long long nxt =
              run + draw_weight<true>(vec_elem<EB>(t, h), vec_elem<EB>(dd, h), kc);
          if (tok < 0 && nxt > target) tok = (int)(e0 + (size_t)(q * VEC + h));
          run = nxt;
        }
      }
    }
    const unsigned int holder = __ballot_sync(0xffffffffu, tok >= 0);
    tok = holder ? __shfl_sync(0xffffffffu, tok, __ffs(holder) - 1) : -1;
    // the buffer goes back to the bulk copies
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  return tok;
}

// Final draw for request b, run by the warp that completed its last R item
// (the chunk sums are in the workspace).
template <int EB, bool PK>
__device__ __noinline__ void final_draw(const Params& P, int b, TempC tc, unsigned char* stage) {
  const int G = P.G, V = P.V, NCR = P.NCR;
  const int lane = threadIdx.x & 31;
  Decision d;
  d.k = 0;
  d.reject = 0;
  d.mt = d.md = d.inv_st = d.rho = 0.0f;
  unsigned int flags = 0;
  {
    // every R item of b read b's decision before arriving, so it is published
    int rb = -1;
    bool ok = false;
    if (lane == 0) {
      const unsigned long long t0 = now_ns();
      while (!(ok = read_record(&P.dec[b], rb, d)) && now_ns() - t0 < P.wait_ns) __nanosleep(64);
    }
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) flags |= SV_STATUS_TIMEOUT;
    d.k = __shfl_sync(0xffffffffu, d.k, 0);
    d.reject = __shfl_sync(0xffffffffu, d.reject, 0);
    d.mt = __shfl_sync(0xffffffffu, d.mt, 0);
    d.md = __shfl_sync(0xffffffffu, d.md, 0);
    d.inv_st = __shfl_sync(0xffffffffu, d.inv_st, 0);
    d.rho = __shfl_sync(0xffffffffu, d.rho, 0);
  }
  d.c_hi = tc.hi;
  d.c_lo = tc.lo;
  const ReqAddr A = req_addr<PK>(P, b);
  const float u_s = sanitize_uniform(P.uniforms[A.uf], flags);
  const int k = d.k < 0 ? 0 : (d.k > G ? G : d.k);
  ResidC kc;
  kc.mt = d.mt; kc.md = d.md; kc.inv_st = d.inv_st; kc.rho = d.rho;
  resid_scales(kc);
  kc.hi = d.c_hi; kc.lo = d.c_lo; kc.reject = (d.reject && k < G) ? 1 : 0;
  const char* trow = P.target + (A.t0 + (size_t)k) * (size_t)V * EB;
  const char* drow = kc.reject ? P.draft + (A.d0 + (size_t)k) * (size_t)V * EB : nullptr;
  unsigned long long* rp = P.resid + (size_t)b * P.stride_ncr;

  int tok = chunk_draw<EB, true>(trow, drow, V, NCR, u_s, kc, rp, stage);
  if (lane == 0) {
    if (tok < 0) {
      flags |= SV_STATUS_INTERNAL;
      tok = V - 1;
    }
    P.out_tokens[(size_t)b * (G + 1) + k] = tok;
    if (flags) atomicOr(P.status, flags);
    P.cnt_r[b] = 0;
    // every R item of b is done: nobody reads the decision again in this call
    atom_store_b128(&P.dec[b].tag_a, make_uint4(0u, 0u, 0u, 0u));
    atom_store_b128(&P.dec[b].tag_b, make_uint4(0u, 0u, 0u, 0u));
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


// An unaligned item's elements copied into its stage buffer (which no copy
// targets), padded with -inf to the whole buffer, so that it is reduced by
// the same code, in the same order, as a copied item: a row's statistics do
// not depend on where the row sits in memory.
template <int EB>
__device__ __noinline__ void stage_unaligned(const Meta& m, char* stage) {
  constexpr int AE = kItemBytes / EB;
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < AE; e += 32) {
    if constexpr (EB == 2) {
      const unsigned short x = e < m.n ? __ldg(reinterpret_cast<const unsigned short*>(m.p0) + e)
                                       : (unsigned short)0xff80u;
      reinterpret_cast<unsigned short*>(stage)[e] = x;
    } else {
      const unsigned int x = e < m.n ? __ldg(reinterpret_cast<const unsigned int*>(m.p0) + e)
                                     : 0xff800000u;
      reinterpret_cast<unsigned int*>(stage)[e] = x;
    }
  }
  __syncwarp();
}

// The tail of a partial copied item (the last chunk of a row) set to -inf, so
// the item routines read whole buffers without bounds checks (a -inf logit
// changes neither a maximum nor a sum of exp2, nor the lowest index of a
// finite maximum).
template <int EB>
__device__ __noinline__ void pad_item_tail(char* stage, int n) {
  const int lane = threadIdx.x & 31;
  const uint4 ninf = neg_inf_vec(EB);
  for (int vi = n * EB / 16 + lane; vi < kItemBytes / 16; vi += 32) sts128(stage + vi * 16, ninf);
  __syncwarp();
}

// A item, sampling: (max, sum of exp2) over the item, in two steps so that a
// caller can refill the buffer in between.  item_load_max reads the whole
// item into registers (the buffer is valid throughout: a partial or unaligned
// item is padded with -inf) and returns its maximum; every loaded value feeds
// the maximum, so the buffer's reads are complete when it returns.
// item_exp_sum then sums 2^((z - max) c) from the registers.
constexpr int kItemWords = kItemBytes / 4 / 32;  // 32-bit words of an item per lane (64)

template <int EB>
__device__ __forceinline__ float item_load_max(const char* stage, uint32_t (&w)[kItemWords]) {
  constexpr int VEC = 16 / EB;
  constexpr int NV = kItemBytes / 16 / 32;  // vectors per lane (16)
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int vi = lane + 32 * j;
    const uint4 v = lds128(stage + vi * 16);
    w[4 * j] = v.x;
    w[4 * j + 1] = v.y;
    w[4 * j + 2] = v.z;
    w[4 * j + 3] = v.w;
  }
  if constexpr (EB == 2) {
    // maximum on the packed bf16 pairs (exact), as a log-depth tree
    uint32_t t[kItemWords / 2];
#pragma unroll
    for (int i = 0; i < kItemWords / 2; ++i) t[i] = bf16x2_max(w[i], w[i + kItemWords / 2]);
#pragma unroll
    for (int width = kItemWords / 4; width >= 1; width >>= 1)
#pragma unroll
      for (int i = 0; i < width; ++i) t[i] = bf16x2_max(t[i], t[i + width]);
    return warp_max(bf16x2_hmax(t[0]));
  } else {
    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
      for (int q = 0; q < VEC; ++q) mq[q & 3] = fmaxf(mq[q & 3], __uint_as_float(w[4 * j + q]));
    return warp_max(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])));
  }
}

// The exponent argument is (z - max) c with c = log2(e)/T rounded to one
// float: the constant's rounding (at most |a| 2^-24) is below ex2.approx's own
// relative error for the terms that carry the sum.  (Chunk combines, the
// decision and the draw weights keep the two-term form.)  It is formed with
// one fused multiply-add, z c + RN(-max c): exact before its one rounding,
// but for the constant delta = max c - RN(max c), the product's rounding
// error, which every term shares.  Each term is thus 2^delta too large, and
// the sum is multiplied by 2^-delta once (|delta| <= 2^-24 |max c|, which
// ex2.approx takes to about 2^-22 relative).  Where max c overflows a float
// (logits beyond about 1e36 at small T) the argument is (z - max) c instead.

// Sum of 2^arg(z) over the item's words held by this lane.
template <int EB, bool FUSED>
__device__ __forceinline__ float item_exp_lane(const uint32_t (&w)[kItemWords], float mx, float c1,
                                               float nmc) {
  constexpr int VEC = 16 / EB;
  constexpr int NV = kItemBytes / 16 / 32;
  if constexpr (EB == 2) {
    // the arguments and the sum on float32 pairs, 8 accumulators
    const unsigned long long nm = f2_pack(nmc, nmc), negm = f2_pack(-mx, -mx);
    const unsigned long long cc = f2_pack(c1, c1);
    unsigned long long acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0ull;
#pragma unroll
    for (int i = 0; i < kItemWords; ++i) {
      const unsigned long long a = FUSED ? f2_fma(bf16x2_to_f2(w[i]), cc, nm)
                                         : f2_mul(f2_add(bf16x2_to_f2(w[i]), negm), cc);
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
    return s0 + s1;
  } else {
    float sq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      float e[VEC];
#pragma unroll
      for (int q = 0; q < VEC; ++q) {
        const float z = __uint_as_float(w[4 * j + q]);
        e[q] = ex2_approx(FUSED ? __fmaf_rn(z, c1, nmc) : __fmul_rn(__fsub_rn(z, mx), c1));
      }
#pragma unroll
      for (int u = VEC; u > 1; u >>= 1)
#pragma unroll
        for (int q = 0; q < u / 2; ++q) e[q] = e[2 * q] + e[2 * q + 1];
      sq[j & 3] += e[0];
    }
    return (sq[0] + sq[1]) + (sq[2] + sq[3]);
  }
}

template <int EB>
__device__ __forceinline__ float item_exp_sum(const uint32_t (&w)[kItemWords], float mx, float c_hi,
                                              float c_lo) {
  if (!(mx > -INFINITY)) return 0.0f;
  const float c1 = __fadd_rn(c_hi, c_lo);
  const float nmc = -__fmul_rn(mx, c1);
  if (fabsf(nmc) <= 3.0e38f) {  // the same on every lane
    const float delta = __fmaf_rn(mx, c1, nmc);  // exact
    return __fmul_rn(warp_sum(item_exp_lane<EB, true>(w, mx, c1, nmc)), ex2_approx(-delta));
  }
  return warp_sum(item_exp_lane<EB, false>(w, mx, c1, nmc));
}

template <int EB>
__device__ __forceinline__ float2 a_item_sample(const Meta& m, const char* stage) {
  uint32_t w[kItemWords];
  const float mx = item_load_max<EB>(stage, w);
  return make_float2(mx, item_exp_sum<EB>(w, mx, m.c_hi, m.c_lo));
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
    // the maximum (independent chains), then the lowest index holding it (a
    // partial item is padded with -inf; the float32 index scan skips the pad)
    const int nvec = m.n / VEC;
    if constexpr (EB == 2) {
      // maximum on the packed pairs as a log-depth tree; a lane holding the
      // warp maximum finds its first vector holding it, then the element
      constexpr int NW = NV * 4;
      uint32_t w[NW];
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int vi = lane + 32 * j;
        const uint4 v = lds128(stage + vi * 16);
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
      v[j] = lds128(stage + vi * 16);
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

// R item: fixed-point sum of the draw weights over the chunk.  bf16 logits
// are processed two at a time in packed float32 pairs, with the same
// operations, in the same order, as draw_x and fix_parts.
template <int EB, bool REJECT>
__device__ __forceinline__ unsigned long long r_item_sum(const Meta& m, const char* stage,
                                                         const ResidC& kc) {
  constexpr int VEC = 16 / EB;
  constexpr int NV = kHalfBytes / 16 / 32;  // vectors per lane per row (8)
  const int lane = threadIdx.x & 31;
  const int nvec = m.n / VEC;
  FixAcc a0{0u, 0u, 0u}, a1{0u, 0u, 0u};  // independent chains
  if constexpr (EB == 2) {
    const unsigned long long negmt = f2_pack(-kc.mt, -kc.mt), negmd = f2_pack(-kc.md, -kc.md);
    const unsigned long long chi = f2_pack(kc.hi, kc.hi), clo = f2_pack(kc.lo, kc.lo);
    const unsigned long long nrho = f2_pack(kc.nrho, kc.nrho), c16 = f2_pack(kc.c16, kc.c16);
    const unsigned long long p23 = f2_pack(8388608.0f, 8388608.0f);
    const unsigned long long n23 = f2_pack(-8388608.0f, -8388608.0f);
    const unsigned long long mone = f2_pack(-1.0f, -1.0f), p16 = f2_pack(65536.0f, 65536.0f);
    const unsigned long long c15 = f2_pack(12582912.0f, 12582912.0f);
#pragma unroll kRUnroll
    for (int j = 0; j < NV; ++j) {
      const int vi = lane + 32 * j;
      if (vi < nvec) {
        const uint4 t = lds128(stage + vi * 16);
        const uint4 d = REJECT ? lds128(stage + kHalfBytes + vi * 16) : t;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const unsigned long long dt = f2_add(bf16x2_to_f2(vec_word(t, q)), negmt);
          float x0, x1;
          f2_unpack(f2_fma(dt, chi, f2_mul(dt, clo)), x0, x1);
          unsigned long long v = f2_pack(ex2_approx(x0), ex2_approx(x1));
          if (REJECT) {
            const unsigned long long dd = f2_add(bf16x2_to_f2(vec_word(d, q)), negmd);
            f2_unpack(f2_fma(dd, chi, f2_mul(dd, clo)), x0, x1);
            const unsigned long long ed = f2_pack(ex2_approx(x0), ex2_approx(x1));
            f2_unpack(f2_fma(ed, nrho, v), x0, x1);
            v = f2_pack(fmaxf(x0, 0.0f), fmaxf(x1, 0.0f));
          }
          const unsigned long long y = f2_mul(v, c16);
          const unsigned long long tt = f2_add(y, p23);
          const unsigned long long dl = f2_fma(f2_add(tt, n23), mone, y);
          const unsigned long long t2 = f2_fma(dl, p16, c15);
          float u0, u1, w0, w1;
          f2_unpack(tt, u0, u1);
          f2_unpack(t2, w0, w1);
          FixAcc& a = (q & 1) ? a1 : a0;
          fix_add_parts(a, u0, w0);
          fix_add_parts(a, u1, w1);
        }
      }
    }
  } else {
#pragma unroll kRUnroll
    for (int j = 0; j < NV; ++j) {
      const int vi = lane + 32 * j;
      if (vi < nvec) {
        const uint4 t = lds128(stage + vi * 16);
        const uint4 d = REJECT ? lds128(stage + kHalfBytes + vi * 16) : t;
#pragma unroll
        for (int q = 0; q < VEC; ++q) {
          const float y = draw_x<REJECT>(vec_elem<EB>(t, q), vec_elem<EB>(d, q), kc);
          if (q & 1) fix_add(a1, y); else fix_add(a0, y);
        }
      }
    }
  }
  return fix_value(a0) + fix_value(a1);
}

template <int EB>
__device__ __forceinline__ unsigned long long r_item(const Meta& m, const char* stage) {
  const int lane = threadIdx.x & 31;
  ResidC kc;
  kc.mt = m.mt; kc.md = m.md; kc.inv_st = m.inv_st; kc.rho = m.rho;
  resid_scales(kc);
  kc.hi = m.c_hi; kc.lo = m.c_lo; kc.reject = m.reject;
  unsigned long long sr = 0;
  if (!m.direct) {
    sr = m.reject ? r_item_sum<EB, true>(m, stage, kc) : r_item_sum<EB, false>(m, stage, kc);
  } else {
    for (int e = lane; e < m.n; e += 32) {
      const float zd = m.reject ? direct_elem<EB>(m, 1, e) : -INFINITY;
      sr += draw_weight(direct_elem<EB>(m, 0, e), zd, kc);
    }
  }
  return warp_sum_u64(sr);
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
  int req, row, c;  // request, row within the request, chunk
  int rows, gb;     // rows of req, and its gamma
};

template <int MODE>
__device__ __forceinline__ int rows_of(const int* rowpre, int b) {
  return rowpre[b + 1] - rowpre[b];
}

// gamma of a request from its row count: sampling requests have 2 gamma + 1
// rows, greedy ones (greedy mode, or temperature 0) gamma + 1.
template <int MODE>
__device__ __forceinline__ int gamma_of(int rows, const TempC* tconst, int b) {
  return (MODE == MODE_SAMPLE && tconst[b].hi != 0.0f) ? (rows - 1) / 2 : rows - 1;
}

// Place the cursor on A item j.
template <int MODE>
__device__ __forceinline__ void cursor_seek(Cursor& k, unsigned int j, const int* rowpre, int B,
                                            int NC, const TempC* tconst) {
  k.j = j;
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
  k.gb = gamma_of<MODE>(k.rows, tconst, lo);
}

// Advance the cursor by one A item (never past the last one's successor).
template <int MODE>
__device__ __forceinline__ void cursor_next(Cursor& k, const int* rowpre, int B, int NC,
                                            const TempC* tconst) {
  ++k.j;
  if (++k.c == NC) {
    k.c = 0;
    if (++k.row == k.rows) {
      k.row = 0;
      if (++k.req < B) {
        k.rows = rows_of<MODE>(rowpre, k.req);
        k.gb = gamma_of<MODE>(k.rows, tconst, k.req);
      }
    }
  }
}

// The A item under the cursor.
template <int EB, int MODE, bool PK>
__device__ __forceinline__ void a_item_at(const Params& P, const Cursor& k, float c_hi,
                                          float c_lo, const int* cbase, Meta& m) {
  constexpr int AE = kItemBytes / EB;
  const int G = P.G, V = P.V;
  const ReqAddr A = addr_from_base<PK>(P, k.req, PK ? cbase[k.req] : 0, k.gb);
  size_t roff;
  const char* base;
  if (k.row <= k.gb) {
    m.pslot = k.row;
    roff = (A.t0 + (size_t)k.row) * (size_t)V;
    base = P.target;
  } else {
    const int i = k.row - k.gb - 1;
    m.pslot = G + 1 + i;
    roff = (A.d0 + (size_t)i) * (size_t)V;
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
template <int EB, bool PK>
__device__ __forceinline__ void fill_r_item(const Params& P, const Decision& d, const int* cbase,
                                            Meta& m) {
  constexpr int RE = kHalfBytes / EB;
  const int G = P.G, V = P.V, req = m.b, c = m.c;
  const ReqAddr A = addr_from_base<PK>(P, req, PK ? cbase[req] : 0, 0);
  const int k = d.k < 0 ? 0 : (d.k > G ? G : d.k);
  const int reject = (d.reject && k < G) ? 1 : 0;
  m.kind = KIND_R;
  m.pslot = k;
  m.reject = reject;
  m.n = min(RE, V - c * RE);
  m.p0 = P.target + ((A.t0 + (size_t)k) * (size_t)V + (size_t)c * RE) * EB;
  m.p1 = reject ? P.draft + ((A.d0 + (size_t)k) * (size_t)V + (size_t)c * RE) * EB : nullptr;
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
template <int EB, int MODE, bool PK>
__global__ void __launch_bounds__(kThreads, 1) verify_kernel(Params P) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  int* rowpre = reinterpret_cast<int*>(dsmem + kWarps * kNB * kItemBytes);  // [B+1]
  // [B] (hi, lo) of log2(e)/T per request (sampling)
  TempC* tconst = reinterpret_cast<TempC*>(rowpre + ((P.B + 2) & ~1));
  // [B] packed layout: each request's first draft row (its sanitised cu[b])
  int* cbase = reinterpret_cast<int*>(tconst + P.B);
  __shared__ __align__(8) uint64_t bar[kWarps][kNB];
  __shared__ Meta meta[kWarps][kNB];     // the item in each buffer
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
      unsigned int fl = 0;
      int gb = 0;
      if constexpr (PK) {
        cbase[b] = packed_base(P, b, gb, fl);
      } else {
        const int g_in = P.gamma ? P.gamma[b] : 0;
        gb = clamp_gamma(g_in, G);
        if (g_in != gb) fl |= SV_STATUS_BAD_GAMMA;
      }
      v = gb + 1;
      if (MODE == MODE_SAMPLE) {
        // temperature 0: this request takes the greedy steps (target rows
        // only); its constants are marked with hi = 0
        const float T = P.temperature[b];
        if (T == 0.0f) {
          tconst[b] = TempC{0.0f, 0.0f};
        } else {
          tconst[b] = temp_consts(sanitize_temperature(T, fl));
          v = 2 * gb + 1;
        }
      }
      if (fl && blockIdx.x == 0) atomicOr(P.status, fl);  // reported once
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

  const unsigned int nA = (unsigned int)rowpre[B] * NC;                        // A items
  const unsigned int nR = MODE == MODE_SAMPLE ? (unsigned int)B * NCR : 0u;  // R items
  const unsigned int nwarps = gridDim.x * kWarps;
  // batches: about 1/kBatchDiv of a warp's share, at most kMaxK A items or
  // kMaxRBatch R items
  const unsigned int K = min((unsigned int)kMaxK, max(1u, nA / (nwarps * kBatchDiv)));
  const unsigned int KR = min(kMaxRBatch, max(1u, nR / (nwarps * kBatchDiv)));
  const unsigned int r_backlog = (unsigned int)(SV_BACKLOG_X4 * nwarps * KR / 4u);

  unsigned char* mybuf = dsmem + (size_t)warp * kNB * kItemBytes;
  uint64_t* mybar = bar[warp];
  Meta* mymeta = meta[warp];

  // ---- Work selection -----------------------------------------------------
  // A items come in a fixed order: the first batch of every warp is fixed by
  // its index, later batches are claimed from next_item asynchronously (the
  // claim for the batch after the current one is started when the current
  // one begins).  R items exist only for decided requests: a deciding warp
  // appends its request to the decision queue, and R batches are claimed
  // from r_next (item i = chunk i % NCR of queue slot i / NCR).  While A
  // items remain, a warp takes R work only when the published, unclaimed R
  // items (an estimate from loads started one batch earlier) exceed a
  // backlog of SV_BACKLOG_X4 / 4 batches per warp.  The default (16 batches)
  // means A items first: the SMs are close to issue-bound during the A pass,
  // and residual work taken earlier lengthens it (measured at every backlog
  // from 0 to 16 batches).
  bool a_done = false;         // lane 0: next_item ran past the A items
  unsigned int a_raw = 0;      // lane 0: result of the pending A claim
  bool a_pending = false;      // lane 0
  unsigned int pf_q = 0, pf_r = 0;  // lane 0: q_tail and r_next loaded one batch ago
  auto claim_a = [&]() {
    a_raw = atomicAdd(P.next_item, K);
    a_pending = true;
  };
  auto prefetch = [&]() {
    if (MODE == MODE_SAMPLE) {
      pf_q = ld_relaxed(P.q_tail);
      pf_r = ld_relaxed(P.r_next);
    }
  };
  unsigned int a_first = (blockIdx.x * kWarps + warp) * K;  // fixed first batch
  if (a_first >= nA) a_first = ~0u;
  if (lane == 0) {
    claim_a();
    prefetch();
  }

  Cursor cur;        // current A batch [cur.j, a_end)
  cur.j = 0;
  unsigned int a_end = 0;
  unsigned int r_i = 0, r_end = 0;  // current R batch [r_i, r_end)
  bool more = true;                 // batches may remain
  bool wait_slot = false;           // the next R item's queue slot is not yet published
  bool r_done = false;              // R claims ran past the last rejected request
  unsigned int issued = 0, processed = 0;
  int dec_p = -1, dec_b = 0;        // queue slot and request whose decision is in dc
  Decision dc;
  dc.k = 0;
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
      fence_acquire();  // the other arrivers' partials are visible from here
      // The most recently consumed buffer is free until the next copy is
      // issued: the follow-up uses it as scratch.
      unsigned char* scratch = mybuf + ((processed + kNB - 1) % kNB) * kItemBytes;
      const int gb = gamma_of<MODE>(rows_of<MODE>(rowpre, b), tconst, b);
      if (pend_kind == KIND_A) {
        if (MODE == MODE_SAMPLE && tconst[b].hi != 0.0f) {
          decide_sample<EB, PK>(P, b, gb, tconst[b], reinterpret_cast<float*>(scratch));
        } else {
          decide_greedy<PK>(P, b, gb, reinterpret_cast<int*>(scratch));
          if (MODE == MODE_SAMPLE && lane == 0) {  // counted like any decision
            __threadfence();
            atomicAdd(P.dec_count, 1u);
          }
        }
      } else {
        final_draw<EB, PK>(P, b, tconst[b], scratch);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
      pend_old = atom_add_release(cnt, acc_n);
    }
    pend_kind = acc_kind;
    pend_b = acc_b;
    acc_n = 0;
  };

  // Fetch the decision in queue slot p into dc (dec_p, dec_b); false while
  // the slot is not yet published.
  auto load_slot = [&](int p) -> bool {
    if (p == dec_p) return true;
    unsigned int ok = 0;
    int b = 0;
    Decision d;
    d.k = d.reject = 0;
    d.mt = d.md = d.inv_st = d.rho = 0.0f;
    if (lane == 0) ok = read_record(&P.queue[p], b, d) ? 1u : 0u;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      dec_b = __shfl_sync(0xffffffffu, b, 0);
      dc.k = __shfl_sync(0xffffffffu, d.k, 0);
      dc.reject = __shfl_sync(0xffffffffu, d.reject, 0);
      dc.mt = __shfl_sync(0xffffffffu, d.mt, 0);
      dc.md = __shfl_sync(0xffffffffu, d.md, 0);
      dc.inv_st = __shfl_sync(0xffffffffu, d.inv_st, 0);
      dc.rho = __shfl_sync(0xffffffffu, d.rho, 0);
      const TempC tc = tconst[dec_b];
      dc.c_hi = tc.hi;
      dc.c_lo = tc.lo;
      dec_p = p;
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

  // lane 0: the next A batch [lo, hi) from the pending claim; false once the
  // A items are all claimed.
  auto take_a = [&](unsigned int& lo, unsigned int& hi) -> bool {
    if (a_done) return false;
    if (!a_pending) claim_a();
    const unsigned long long j = (unsigned long long)nwarps * K + a_raw;
    a_pending = false;
    if (j >= nA) {
      a_done = true;
      return false;
    }
    lo = (unsigned int)j;
    hi = min(lo + K, nA);
    claim_a();  // the batch after this one
    return true;
  };

  // Choose the next batch at a batch boundary.  0: none left, 1: A, 2: R.
  auto next_batch = [&]() -> int {
    unsigned int kind = 0, lo = 0, hi = 0;
    if (lane == 0) {
      if (a_first != ~0u) {  // the fixed first batch
        kind = 1;
        lo = a_first;
        hi = min(a_first + K, nA);
        a_first = ~0u;
      }
      // R work while A items remain only if the published, unclaimed R items
      // (as loaded a batch ago) exceed a backlog of SV_BACKLOG_X4 / 4 batches
      // per warp (16 by default, so in practice A items first): A items gate
      // the decisions, and the R work left when they run out is spread over
      // every warp.
      if (kind == 0 && MODE == MODE_SAMPLE && !r_done && pf_r < nR &&
          (a_done ? pf_r < pf_q * (unsigned int)NCR
                  : pf_r + r_backlog < pf_q * (unsigned int)NCR)) {
        const unsigned int i = atomicAdd(P.r_next, KR);
        if (i < nR) {
          kind = 2;
          lo = i;
          hi = min(i + KR, nR);
        }
      }
      if (kind == 0 && take_a(lo, hi)) kind = 1;
      // no A items left: R items not yet published are claimed too (their
      // slots are waited for once this warp's pipeline is drained)
      if (kind == 0 && MODE == MODE_SAMPLE && !r_done) {
        const unsigned int i = atomicAdd(P.r_next, KR);
        if (i < nR) {
          kind = 2;
          lo = i;
          hi = min(i + KR, nR);
        }
      }
      prefetch();
    }
    kind = __shfl_sync(0xffffffffu, kind, 0);
    lo = __shfl_sync(0xffffffffu, lo, 0);
    hi = __shfl_sync(0xffffffffu, hi, 0);
    if (kind == 1) {
      cursor_seek<MODE>(cur, lo, rowpre, B, NC, tconst);
      a_end = hi;
    } else if (kind == 2) {
      r_i = lo;
      r_end = hi;
    }
    return (int)kind;
  };

  while (!failed) {
    // 1. keep kNB copies in flight
    while (!wait_slot && issued - processed < (unsigned int)kNB) {
      if (cur.j == a_end && r_i == r_end) {
        if (!more || next_batch() == 0) {
          more = false;
          break;
        }
      }
      if (cur.j < a_end) {
        Meta a;
        if (MODE == MODE_SAMPLE) {
          const TempC tc = tconst[cur.req];
          a_item_at<EB, MODE, PK>(P, cur, tc.hi, tc.lo, cbase, a);
        } else {
          a_item_at<EB, MODE, PK>(P, cur, 0.0f, 0.0f, cbase, a);
        }
        issue(a);
        cursor_next<MODE>(cur, rowpre, B, NC, tconst);
      } else if (MODE == MODE_SAMPLE) {
        if (!load_slot((int)(r_i / (unsigned int)NCR))) {
          wait_slot = true;  // decided soon: wait once the pipeline is drained
          break;
        }
        Meta r;
        r.b = dec_b;
        r.c = (int)(r_i % (unsigned int)NCR);
        fill_r_item<EB, PK>(P, dc, cbase, r);
        issue(r);
        ++r_i;
      }
    }

    // 2. process the oldest item in flight
    if (issued != processed) {
      const int s = (int)(processed % kNB);
      if (!mbar_wait(&mybar[s], (processed / kNB) & 1u, P.wait_ns)) {
        flags |= SV_STATUS_TIMEOUT;
        failed = true;
        break;
      }
      const Meta& m = mymeta[s];
      const int m_kind = m.kind, m_b = m.b;
      char* stage = reinterpret_cast<char*>(mybuf + s * kItemBytes);
      if (m_kind == KIND_A) {
        const bool staged = MODE == MODE_SAMPLE && m.c_hi != 0.0f;
        const bool padded = !m.direct && m.n < kItemBytes / EB;  // a row's last chunk
        if (staged && m.direct) stage_unaligned<EB>(m, stage);
        else if (padded) pad_item_tail<EB>(stage, m.n);
        const float2 part = staged ? a_item_sample<EB>(m, stage) : a_item_greedy<EB>(m, stage);
        if (lane == 0) P.stats[((size_t)m_b * (2 * G + 1) + m.pslot) * P.stride_nc + m.c] = part;
        // stores into the buffer are ordered before the next bulk copy into it
        if ((staged && m.direct) || padded) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      } else {
        const unsigned long long part = r_item<EB>(m, stage);
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
    if (wait_slot) {
      // While A items remain, do those first (the R batch is kept): a warp
      // never waits while A work that a decision may need is unclaimed.
      unsigned int got = 0, lo = 0, hi = 0;
      if (lane == 0) got = take_a(lo, hi) ? 1u : 0u;
      if (__shfl_sync(0xffffffffu, got, 0)) {
        lo = __shfl_sync(0xffffffffu, lo, 0);
        hi = __shfl_sync(0xffffffffu, hi, 0);
        cursor_seek<MODE>(cur, lo, rowpre, B, NC, tconst);
        a_end = hi;
        wait_slot = false;
        continue;
      }
      // Publish held arrivals (a decision may depend on them), then wait for
      // the queue slot of the next R item.
      flush();
      settle();
      // Requests whose drafts were all accepted have no R work and no queue
      // slot: once every request is decided, a slot at or past the queue's
      // end never comes and the batch is void.
      const int p = (int)(r_i / (unsigned int)NCR);
      int state = 0;
      if (lane == 0) {
        const unsigned long long t0 = now_ns();
        unsigned int ns = 64;
        while (!(ld_acquire(&P.queue[p].tag_a) & kDecTag)) {
          if (ld_acquire(P.dec_count) == (unsigned int)B && (unsigned int)p >= ld_acquire(P.q_tail)) {
            state = 2;
            break;
          }
          if (now_ns() - t0 > P.wait_ns) {
            state = 1;
            break;
          }
          __nanosleep(ns);
          ns = ns < 1024 ? 2 * ns : ns;
        }
      }
      state = __shfl_sync(0xffffffffu, state, 0);
      if (state == 1) {
        flags |= SV_STATUS_TIMEOUT;
        failed = true;
        break;
      }
      wait_slot = false;  // the record is complete shortly after its tag
      if (state == 2) {   // no R work left
        r_i = r_end;
        r_done = true;
      }
      continue;
    }
    if (!more) break;  // all work done
  }

  // No copy may still be landing in this warp's buffers when it leaves.
  if (failed) {
    for (unsigned int p = processed; p < issued; ++p)
      (void)mbar_wait(&mybar[p % kNB], (p / kNB) & 1u, P.wait_ns);
  } else {
    flush();
    settle();
  }
  if (lane == 0 && flags) atomicOr(P.status, flags);
  __syncthreads();
  // the last CTA out resets the claim counters and the queue for the next call
  if (tid == 0) {
    __threadfence();
    sh_last = atomicAdd(P.exit_count, 1u) == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (sh_last) {
    if (tid == 0) {
      *P.next_item = 0;
      *P.r_next = 0;
      *P.q_tail = 0;
      *P.dec_count = 0;
      *P.exit_count = 0;
    }
    if (MODE == MODE_SAMPLE)
      for (int p = tid; p < B; p += kThreads) {
        P.queue[p].tag_a = 0u;
        P.queue[p].tag_b = 0u;
      }
    __threadfence();
  }
}

// ---------------------------------------------------------------------------
// Small batches: one thread-block cluster per request
// ---------------------------------------------------------------------------
// With few requests the persistent schedule is bound by its chain of
// global-memory synchronisations (arrival counters, decision records, queue
// polls), each an L2 round trip.  Here request b gets cluster b of C CTAs,
// one per SM.  Every warp streams a fixed share of the request's A items and
// stores each partial into the shared memory of every CTA of the cluster; a
// cluster barrier replaces the arrival counter; each CTA's warp 0 then
// computes the decision from its own copy (the arithmetic of the persistent
// path; the leader, rank 0, writes the outputs).  Each warp keeps its unit (a
// target chunk and the draft chunk of the same position) in its two staging
// buffers; after a reject the CTAs compute the residual block sums of the
// rejected row from those buffers, exchange their totals, and after a second
// barrier the CTA holding floor(u S) walks one resident block of 256 (bf16)
// or 128 (float32) tokens.
constexpr int kClusterMax = 16;                  // CTAs per cluster, at most
constexpr int kBlk = 8;                          // blocks per R item: one per vector column
constexpr int kClusterTables = 24 * 1024;        // partials, fallback block sums, decision
constexpr size_t kClusterSmem = (size_t)kWarps * kNB * kItemBytes + kClusterTables;
// about 5 KB of static shared memory (barriers, item records, unit block sums)
static_assert(kClusterSmem + 6 * 1024 <= 227 * 1024, "cluster shared memory budget");

struct ClusterDec {  // the decision, as every CTA of the cluster holds it
  int k, go;         // go: 1 when R items follow (a rejected draft)
  float mt, md, inv_st, rho, c_hi, c_lo;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: stores before it (shared memory
// of any CTA) are visible to loads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of location p in CTA `rank`.
__device__ __forceinline__ uint32_t rank_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f2(uint32_t a, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ void st_cluster_u64(uint32_t a, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

// Residual draw weights of a resident unit (a target chunk and the draft
// chunk of the same position, each AE logits in its own staging buffer),
// summed per block of 32 vectors: blk[j] is block j0 + j, whose vector l + 32
// (j0 + j) lane l reads, as round(w 2^39) with the per-token operations of
// draw_weight (a block's sum therefore equals the prefix walk over it).
// Four per-lane values reduced over the warp at once: after the exchanges
// with lanes 16 and 8 apart each lane holds partial sums of one value (the
// value index is lane bits 4..3), then three butterfly steps finish them.
// Returns value (lane >> 3) & 3 on every lane.
__device__ __forceinline__ unsigned long long warp_sum4_u64(const unsigned long long (&v)[4]) {
  const int lane = threadIdx.x & 31;
  const bool hi16 = (lane & 16) != 0, hi8 = (lane & 8) != 0;
  // step 1: lanes 0-15 keep values 0, 1; lanes 16-31 keep values 2, 3
  unsigned long long a0 = hi16 ? v[2] : v[0], a1 = hi16 ? v[3] : v[1];
  const unsigned long long s0 = hi16 ? v[0] : v[2], s1 = hi16 ? v[1] : v[3];
  a0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  a1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  // step 2: within each half, lanes with bit 3 clear keep the first value
  unsigned long long a = hi8 ? a1 : a0;
  a += __shfl_xor_sync(0xffffffffu, hi8 ? a0 : a1, 8);
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
  return a;
}

template <int EB, int NJ>
__device__ __forceinline__ void unit_blocks(const char* tb, const char* db, int nvec, int j0,
                                            const ResidC& kc, unsigned long long (&blk)[NJ]) {
  static_assert(NJ == 4, "blocks are reduced four at a time");
  constexpr int VEC = 16 / EB;
  const int lane = threadIdx.x & 31;
  unsigned long long own[NJ];
  if constexpr (EB == 2) {
    // packed pairs: the operations of r_item_sum
    const unsigned long long negmt = f2_pack(-kc.mt, -kc.mt), negmd = f2_pack(-kc.md, -kc.md);
    const unsigned long long chi = f2_pack(kc.hi, kc.hi), clo = f2_pack(kc.lo, kc.lo);
    const unsigned long long nrho = f2_pack(kc.nrho, kc.nrho), c16 = f2_pack(kc.c16, kc.c16);
    const unsigned long long p23 = f2_pack(8388608.0f, 8388608.0f);
    const unsigned long long n23 = f2_pack(-8388608.0f, -8388608.0f);
    const unsigned long long mone = f2_pack(-1.0f, -1.0f), p16 = f2_pack(65536.0f, 65536.0f);
    const unsigned long long c15 = f2_pack(12582912.0f, 12582912.0f);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int vi = lane + 32 * (j0 + j);
      FixAcc a{0u, 0u, 0u};
      if (vi < nvec) {
        const uint4 t = lds128(tb + vi * 16);
        const uint4 d = lds128(db + vi * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const unsigned long long dt = f2_add(bf16x2_to_f2(vec_word(t, q)), negmt);
          float x0, x1;
          f2_unpack(f2_fma(dt, chi, f2_mul(dt, clo)), x0, x1);
          const unsigned long long v0 = f2_pack(ex2_approx(x0), ex2_approx(x1));
          const unsigned long long dd = f2_add(bf16x2_to_f2(vec_word(d, q)), negmd);
          f2_unpack(f2_fma(dd, chi, f2_mul(dd, clo)), x0, x1);
          const unsigned long long ed = f2_pack(ex2_approx(x0), ex2_approx(x1));
          f2_unpack(f2_fma(ed, nrho, v0), x0, x1);
          const unsigned long long v = f2_pack(fmaxf(x0, 0.0f), fmaxf(x1, 0.0f));
          const unsigned long long y = f2_mul(v, c16);
          const unsigned long long tt = f2_add(y, p23);
          const unsigned long long dl = f2_fma(f2_add(tt, n23), mone, y);
          const unsigned long long t2 = f2_fma(dl, p16, c15);
          float u0, u1, w0, w1;
          f2_unpack(tt, u0, u1);
          f2_unpack(t2, w0, w1);
          fix_add_parts(a, u0, w0);
          fix_add_parts(a, u1, w1);
        }
      }
      own[j] = fix_value(a);
    }
  } else {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int vi = lane + 32 * (j0 + j);
      FixAcc a{0u, 0u, 0u};
      if (vi < nvec) {
        const uint4 t = lds128(tb + vi * 16);
        const uint4 d = lds128(db + vi * 16);
#pragma unroll
        for (int q = 0; q < VEC; ++q)
          fix_add(a, draw_x<true>(vec_elem<EB>(t, q), vec_elem<EB>(d, q), kc));
      }
      own[j] = fix_value(a);
    }
  }
  const unsigned long long r = warp_sum4_u64(own);
#pragma unroll
  for (int q = 0; q < NJ; ++q) blk[q] = __shfl_sync(0xffffffffu, r, 8 * q);
}

// Block sums of the draw weights of target row k alone (kc.reject == 0), for
// the fallback when the residual vanished in fixed point: block bl, warp by
// warp over the leader CTA, each lane one vector read from global memory.
template <int EB>
__device__ __noinline__ void p_blocks(const char* trow, int V, const ResidC& kc, int nblk,
                                      unsigned long long* blk) {
  constexpr int VEC = 16 / EB;
  constexpr int RE = kHalfBytes / EB;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int bl = warp; bl < nblk; bl += kWarps) {
    const int c = bl / kBlk, j = bl % kBlk;
    const size_t e0 = (size_t)c * RE + (size_t)(lane + 32 * j) * VEC;
    unsigned long long s = 0;
#pragma unroll
    for (int h = 0; h < VEC; ++h) {
      const size_t e = e0 + (size_t)h;
      if (e < (size_t)V) s += draw_weight<false>(load_elem<EB>(trow, e), -INFINITY, kc);
    }
    s = warp_sum_u64(s);
    if (lane == 0) blk[bl] = s;
  }
}

// Final draw on the cluster path (leader warp 0): the block whose prefix
// passes floor(u S), then one pass over its tokens, one vector per lane.
template <int EB>
__device__ __noinline__ int cluster_walk(const char* trow, const char* drow, int V, float u_s,
                                         const ResidC& kc, const unsigned long long* blk,
                                         int nblk, unsigned int& flags) {
  constexpr int VEC = 16 / EB;
  constexpr int RE = kHalfBytes / EB;
  const int lane = threadIdx.x & 31;
  // 1. the block: lane l owns blocks [b0, b1); then the blocks of the lane
  //    holding floor(u S) are scanned 32 at a time
  const int bpl = (nblk + 31) >> 5;
  const int b0 = min(nblk, lane * bpl), b1 = min(nblk, b0 + bpl);
  unsigned long long own = 0;
#pragma unroll 4
  for (int bl = b0; bl < b1; ++bl) own += blk[bl];
  const unsigned long long incl = warp_incl_scan_u64(own);
  const unsigned long long S = __shfl_sync(0xffffffffu, incl, 31);
  const unsigned long long target = scaled_target(u_s, S);  // < S
  int bs = -1;
  unsigned long long base = 0;
  {
    const unsigned long long excl = incl - own;
    const unsigned int hit = __ballot_sync(0xffffffffu, excl <= target && target < incl);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const int lo = __shfl_sync(0xffffffffu, b0, l), hi = __shfl_sync(0xffffffffu, b1, l);
      base = __shfl_sync(0xffffffffu, excl, l);
#pragma unroll 1
      for (int g0 = lo; g0 < hi && bs < 0; g0 += 32) {
        const int bl = g0 + lane;
        const unsigned long long v = bl < hi ? blk[bl] : 0ull;
        const unsigned long long vi = warp_incl_scan_u64(v);
        const unsigned long long ve = vi - v;
        const unsigned int h2 =
            __ballot_sync(0xffffffffu, bl < hi && base + ve <= target && target < base + vi);
        if (h2) {
          const int l2 = __ffs(h2) - 1;
          bs = g0 + l2;
          base += __shfl_sync(0xffffffffu, ve, l2);
        } else {
          base += __shfl_sync(0xffffffffu, vi, 31);
        }
      }
    }
  }
  if (bs < 0) {
    flags |= SV_STATUS_INTERNAL;
    return V - 1;
  }
  // 2. the token inside block bs: lane l holds tokens [e0, e0 + VEC)
  const size_t e0 = (size_t)(bs / kBlk) * RE + (size_t)(lane + 32 * (bs % kBlk)) * VEC;
  float zt[VEC], zd[VEC];
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(trow) | reinterpret_cast<uintptr_t>(drow)) & 15) == 0 &&
                      e0 + VEC <= (size_t)V;
  if (vec_ok) {
    const uint4 t = __ldcg(reinterpret_cast<const uint4*>(trow + e0 * EB));
    const uint4 d = drow ? __ldcg(reinterpret_cast<const uint4*>(drow + e0 * EB)) : neg_inf_vec(EB);
#pragma unroll
    for (int h = 0; h < VEC; ++h) {
      zt[h] = vec_elem<EB>(t, h);
      zd[h] = vec_elem<EB>(d, h);
    }
  } else {
#pragma unroll
    for (int h = 0; h < VEC; ++h) {
      const size_t e = e0 + (size_t)h;
      zt[h] = e < (size_t)V ? load_elem<EB>(trow, e) : -INFINITY;
      zd[h] = (drow && e < (size_t)V) ? load_elem<EB>(drow, e) : -INFINITY;
    }
  }
  unsigned long long w[VEC];
  unsigned long long lsum = 0;
#pragma unroll
  for (int h = 0; h < VEC; ++h) {
    w[h] = draw_weight(zt[h], zd[h], kc);
    lsum += w[h];
  }
  const unsigned long long li = warp_incl_scan_u64(lsum);
  unsigned long long run = base + li - lsum;
  int tok = -1;
  if (run <= target && target < run + lsum) {
#pragma unroll
    for (int h = 0; h < VEC; ++h) {
      if (tok < 0 && run + w[h] > target) tok = (int)(e0 + (size_t)h);
      run += w[h];
    }
  }
  const unsigned int holder = __ballot_sync(0xffffffffu, tok >= 0);
  if (!holder) {
    flags |= SV_STATUS_INTERNAL;
    return V - 1;
  }
  return __shfl_sync(0xffffffffu, tok, __ffs(holder) - 1);
}

// One request per cluster, each warp at most one unit of the request's A
// work: unit u = c (gamma_b + 1) + i is chunk c of target row i and, for a
// sampling position i < gamma_b, chunk c of draft row i (kept in the warp's
// two staging buffers to the end).  Shared memory: the buffers, then (the
// same layout in every CTA) the partials [2G+1][NC], the leader's block sums
// for the vanished-residual fallback [NCR][kBlk], the block sums of this
// CTA's residual units [kWarps][kUnitBlk], the CTAs' residual totals [C] and
// the decision.
constexpr int kUnitBlk = 2 * kBlk;  // blocks per unit (an A chunk is two R chunks)

template <int EB, int MODE, bool PK>
__global__ void __launch_bounds__(kThreads, 1) cluster_kernel(Params P) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ __align__(8) uint64_t bar[kWarps][kNB];
  __shared__ Meta cmeta[kWarps][kNB];  // the item in each buffer
  __shared__ unsigned long long ublk[kWarps][kUnitBlk];
  __shared__ unsigned long long tot[kClusterMax];
  __shared__ unsigned long long cta_sum;  // this CTA's residual total
  __shared__ int sh_pick;
  __shared__ float rsbuf[192];  // the decision's row statistics
  constexpr int AE = kItemBytes / EB;   // logits per A item
  constexpr int VEC = 16 / EB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_size();
  const int b = (int)cluster_index();
  const int G = P.G, V = P.V, NC = P.NC, NCR = P.NCR;
  float2* part = reinterpret_cast<float2*>(dsmem + (size_t)kWarps * kNB * kItemBytes);
  unsigned long long* blk = reinterpret_cast<unsigned long long*>(part + (size_t)(2 * G + 1) * NC);
  ClusterDec* cdec = reinterpret_cast<ClusterDec*>(blk + (size_t)NCR * kBlk);
  unsigned char* mybuf = dsmem + (size_t)warp * kNB * kItemBytes;
  uint64_t* mybar = bar[warp];
  Meta* mymeta = cmeta[warp];

  const unsigned int gw = rank * kWarps + (unsigned int)warp;
  // Units: u = c (G + 1) + i is chunk c of target row i and, for a sampling
  // position i < G, chunk c of draft row i; units of rows past gamma_b are
  // void.  Warp gw holds unit gw (the host checks (G + 1) NC <= C kWarps).
  const int per = G + 1;
  auto unit_row = [&](unsigned int u) { return (int)(u % (unsigned int)per); };
  auto unit_chunk = [&](unsigned int u) { return (int)(u / (unsigned int)per); };
  const unsigned int nU = (unsigned int)per * (unsigned int)NC;
  const bool has = gw < nU;
  const int ui = has ? unit_row(gw) : 0, uc = has ? unit_chunk(gw) : 0;
  const int un = min(AE, V - uc * AE);  // logits in the unit's chunk
  // padded layout: rows 0..G of target and 0..G-1 of draft exist for every
  // request, so the unit's copies may start before gamma_b is known
  int nitem = !has ? 0 : (MODE == MODE_SAMPLE && ui < G ? 2 : 1);

  // Each warp's lane 0 readies its own barriers, so its copies can start at
  // once: in the padded layout a unit's rows do not depend on gamma_b, and the
  // target chunk goes to buffer 0, the draft chunk (sampling) to buffer 1 before
  // the request's values are read.  A copy of a row that turns out void is still
  // waited for, then ignored.  In the packed layout the rows past gamma_b
  // belong to other requests (or lie past the arrays), so the copies wait for
  // cu_draft and cover rows up to gamma_b only.
  auto issue_unit = [&](const ReqAddr& R) {
    for (int h = 0; h < nitem; ++h) {
      Meta m;
      m.kind = KIND_A;
      m.pslot = h ? G + 1 + ui : ui;
      m.c = uc;
      m.n = un;
      const size_t row = h ? R.d0 + (size_t)ui : R.t0 + (size_t)ui;
      m.p0 = (h ? P.draft : P.target) + (row * (size_t)V + (size_t)uc * AE) * EB;
      m.p1 = nullptr;
      m.direct = ((reinterpret_cast<uintptr_t>(m.p0) & 15) != 0 || ((m.n * EB) & 15) != 0) ? 1 : 0;
      if (lane == 0) {
        mymeta[h] = m;
        if (m.direct) {
          mbar_arrive(&mybar[h]);
        } else {
          mbar_arrive_expect_tx(&mybar[h], (unsigned int)(m.n * EB));
          bulk_copy_g2s(mybuf + h * kItemBytes, m.p0, (unsigned int)(m.n * EB), &mybar[h]);
        }
      }
    }
    __syncwarp();
  };
  if (lane == 0) {
    for (int s = 0; s < kNB; ++s) mbar_init(&mybar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if constexpr (!PK) issue_unit(addr_from_base<false>(P, b, 0, 0));

  // the request: draft length, addresses, temperature constants
  unsigned int rflags = 0, flags = 0;
  int gb = 0, base = 0;
  if constexpr (PK) {
    base = packed_base(P, b, gb, rflags);
  } else {
    const int g_in = P.gamma ? P.gamma[b] : 0;
    gb = clamp_gamma(g_in, G);
    if (g_in != gb) rflags |= SV_STATUS_BAD_GAMMA;
  }
  const ReqAddr A = addr_from_base<PK>(P, b, base, gb);
  if constexpr (PK) {
    nitem = (!has || ui > gb) ? 0 : (MODE == MODE_SAMPLE && ui < gb ? 2 : 1);
    issue_unit(A);
  }
  bool greedy = MODE == MODE_GREEDY;
  TempC tc{0.0f, 0.0f};
  if (MODE == MODE_SAMPLE) {
    const float T = P.temperature[b];
    if (T == 0.0f) greedy = true;  // this request takes the greedy steps
    else tc = temp_consts(sanitize_temperature(T, rflags));
  }
  const bool sample = MODE == MODE_SAMPLE && !greedy;
  if (tid == 0) cta_sum = 0ull;
  __syncthreads();
  // every CTA decides: its warp 0 requests the draft inputs and the final
  // draw's uniform before its items
  DraftIn gin{0, 0.0f, 0.0f, 0.0f, 0u};
  float u_fin = 0.0f;
  unsigned int uflags = 0;
  if (sample && warp == 0) {
    gin = gather_drafts<EB>(P, A, gb);
    u_fin = sanitize_uniform(P.uniforms[A.uf], uflags);
  }

  // ---- this warp's A items: the target chunk of row ui <= gamma_b and, for a
  // sampling position ui < gamma_b, its draft chunk
  bool failed = false;
  {
    const int use = ui > gb ? 0 : (sample && ui < gb ? 2 : 1);  // items that count
    // lane r < C stores each partial into CTA r: every CTA decides locally
    const uint32_t part_r = rank_addr(part, (uint32_t)lane < C ? (uint32_t)lane : 0u);
    for (int h = 0; h < nitem; ++h) {  // every copy is waited for (bounded)
      if (!mbar_wait(&mybar[h], 0u, P.wait_ns)) {
        flags |= SV_STATUS_TIMEOUT;
        failed = true;
      }
      if (h < use) {
        // An item that could not be read still stores a (NaN, 0) partial, so
        // every CTA holds the same table and takes the same branches below.
        float2 pr = make_float2(NAN, 0.0f);
        if (!failed) {
          if (lane == 0) {  // the temperature constants are known by now
            mymeta[h].c_hi = tc.hi;
            mymeta[h].c_lo = tc.lo;
          }
          __syncwarp();
          const Meta& m = mymeta[h];
          char* stage = reinterpret_cast<char*>(mybuf + h * kItemBytes);
          if (sample && m.direct) stage_unaligned<EB>(m, stage);
          else if (!m.direct && m.n < AE) pad_item_tail<EB>(stage, m.n);
          pr = sample ? a_item_sample<EB>(m, stage) : a_item_greedy<EB>(m, stage);
        }
        const Meta& m = mymeta[h];
        if ((uint32_t)lane < C)
          st_cluster_f2(part_r + (uint32_t)((m.pslot * NC + m.c) * (int)sizeof(float2)), pr);
      }
      __syncwarp();
    }
  }
  cluster_sync();  // every CTA holds every partial

  // ---- the decision: the leader's warp 0 writes the outputs; in sampling
  // mode every other CTA's warp 0 computes the same decision from its own
  // copy of the partials (identical data, identical arithmetic)
  if (greedy && rank != 0) return;  // greedy: no further cluster work
  if (warp == 0) {
    float* rs = rsbuf;
    const SharedParts sp{part, NC};
    ClusterDec cd;
    cd.k = 0;
    cd.go = 0;
    cd.mt = cd.md = cd.inv_st = cd.rho = 0.0f;
    cd.c_hi = tc.hi;
    cd.c_lo = tc.lo;
    if (greedy) {
      greedy_core<PK>(P, sp, b, gb, reinterpret_cast<int*>(rs));
    } else {
      Decision d;
      d.k = 0;
      d.reject = 0;
      d.mt = d.md = d.inv_st = d.rho = 0.0f;
      const int k = decide_core<EB, PK>(P, sp, b, gb, tc, rs, A, gin, d, rank == 0);
      cd.k = k;
      cd.go = __shfl_sync(0xffffffffu, d.reject, 0);
      cd.mt = __shfl_sync(0xffffffffu, d.mt, 0);
      cd.md = __shfl_sync(0xffffffffu, d.md, 0);
      cd.inv_st = __shfl_sync(0xffffffffu, d.inv_st, 0);
      cd.rho = __shfl_sync(0xffffffffu, d.rho, 0);
      // every draft accepted: no residual pass follows, so this warp's
      // buffers are free for the bonus draw's staging
      if (k == gb && rank == 0) final_bonus<EB, PK>(P, sp, b, gb, tc, rs[gb], mybuf);
    }
    if (lane == 0) {
      *cdec = cd;
      if (rank == 0 && rflags) atomicOr(P.status, rflags);
    }
  }
  __syncthreads();  // the CTA's warps see its decision
  const ClusterDec cd = *cdec;

  if (cd.go) {
    // ---- residual block sums of the rejected position k, from the resident
    // units of row k in this CTA; four warps share a unit
    ResidC kc;
    kc.mt = cd.mt; kc.md = cd.md; kc.inv_st = cd.inv_st; kc.rho = cd.rho;
    resid_scales(kc);
    kc.hi = cd.c_hi; kc.lo = cd.c_lo; kc.reject = 1;
    const int k = cd.k < 0 ? 0 : (cd.k > G ? G : cd.k);
    constexpr int kGroup = 4;                     // blocks per task
    constexpr int kTasks = kUnitBlk / kGroup;     // tasks per unit
    // the CTA's units of row k: warp w holds unit rank kWarps + w, so they
    // sit at warps w0, w0 + per, ... (ku(m) below)
    const int w0 = (int)(((unsigned int)k + (unsigned int)per - (rank * kWarps) % (unsigned int)per) %
                         (unsigned int)per);
    int nk = 0;
    for (int w = w0; w < kWarps && rank * kWarps + (unsigned int)w < nU; w += per) ++nk;
    auto ku = [&](int m) { return w0 + m * per; };
    for (int t = warp; t < nk * kTasks && !failed; t += kWarps) {
      const int w = ku(t / kTasks), g = t % kTasks;
      const unsigned int u = rank * kWarps + (unsigned int)w;
      const int n = min(AE, V - unit_chunk(u) * AE);
      const unsigned char* wb = dsmem + (size_t)w * kNB * kItemBytes;
      unsigned long long bs[kGroup];
      unit_blocks<EB, kGroup>(reinterpret_cast<const char*>(wb),
                              reinterpret_cast<const char*>(wb + kItemBytes), (n + VEC - 1) / VEC,
                              g * kGroup, kc, bs);
#pragma unroll
      for (int j = 0; j < kGroup; ++j)
        if (lane == j) ublk[w][g * kGroup + j] = bs[j];
      if (lane == 0) atomicAdd(&cta_sum, bs[0] + bs[1] + bs[2] + bs[3]);
    }
    __syncthreads();
    // this CTA's residual total into every CTA
    if (warp == 0 && (uint32_t)lane < C) st_cluster_u64(rank_addr(&tot[rank], (uint32_t)lane), cta_sum);
    cluster_sync();  // every CTA holds every CTA's total

    // ---- the final draw.  Units ascend with rank, so the CTAs' totals in
    // rank order are consecutive pieces of row k's residual CDF: the CTA whose
    // piece holds floor(u S) walks its own resident block.
    unsigned long long S = 0, before = 0;
    if (warp == 0) {
      const unsigned long long v = (uint32_t)lane < C ? tot[lane] : 0ull;
      const unsigned long long incl = warp_incl_scan_u64(v);
      S = __shfl_sync(0xffffffffu, incl, 31);
      int pick = -1;
      if (S != 0ull) {
        float uf = u_fin;
        const unsigned long long target = scaled_target(uf, S);
        const unsigned int hit = __ballot_sync(0xffffffffu, (uint32_t)lane < C && incl - v <= target &&
                                                            target < incl);
        pick = hit ? __ffs(hit) - 1 : -2;
        if (pick >= 0) before = __shfl_sync(0xffffffffu, incl - v, pick);
      }
      if (lane == 0) sh_pick = pick;
    }
    __syncthreads();
    const int pick = sh_pick;  // -1: the residual vanished; -2: internal error
    if (pick == -1 && rank == 0) {
      // The residual vanished in fixed point (p_k and q_k agree within its
      // resolution): draw from p_k instead, its block sums computed by the
      // whole leader CTA from global memory.
      kc.reject = 0;
      const int nblk = NCR * kBlk;
      const char* trow = P.target + (A.t0 + (size_t)k) * (size_t)V * EB;
      p_blocks<EB>(trow, V, kc, nblk, blk);
      __syncthreads();
      if (warp == 0) {
        unsigned int wf = uflags;
        const int tok = cluster_walk<EB>(trow, nullptr, V, u_fin, kc, blk, nblk, wf);
        if (lane == 0) {
          P.out_tokens[(size_t)b * (G + 1) + k] = tok;
          flags |= wf;
        }
      }
    } else if (pick == -2 && rank == 0 && warp == 0) {
      flags |= SV_STATUS_INTERNAL;
      if (lane == 0) P.out_tokens[(size_t)b * (G + 1) + k] = V - 1;
    } else if (pick == (int)rank && warp == 0) {
      // the block: this CTA's units of row k in order, 16 blocks each
      const unsigned long long target = scaled_target(u_fin, S);
      int bsel = -1;
      unsigned long long run = before;
#pragma unroll 1
      for (int g0 = 0; g0 < nk * kUnitBlk && bsel < 0; g0 += 32) {
        const int e = g0 + lane;
        const unsigned long long v = e < nk * kUnitBlk ? ublk[ku(e / kUnitBlk)][e % kUnitBlk] : 0ull;
        const unsigned long long vi = warp_incl_scan_u64(v);
        const unsigned long long ve = vi - v;
        const unsigned int h2 = __ballot_sync(0xffffffffu, e < nk * kUnitBlk && run + ve <= target &&
                                                               target < run + vi);
        if (h2) {
          const int l2 = __ffs(h2) - 1;
          bsel = g0 + l2;
          run += __shfl_sync(0xffffffffu, ve, l2);
        } else {
          run += __shfl_sync(0xffffffffu, vi, 31);
        }
      }
      int tok = V - 1;
      if (bsel < 0) {
        flags |= SV_STATUS_INTERNAL;
      } else {
        // the token: lane l holds the block's vector l (tokens e0 .. e0 + VEC - 1)
        const int w = ku(bsel / kUnitBlk), J = bsel % kUnitBlk;
        const unsigned int u = rank * kWarps + (unsigned int)w;
        const int n = min(AE, V - unit_chunk(u) * AE);
        const int vi = lane + 32 * J;
        const unsigned char* wb = dsmem + (size_t)w * kNB * kItemBytes;
        const uint4 t = vi < (n + VEC - 1) / VEC ? lds128(wb + vi * 16) : neg_inf_vec(EB);
        const uint4 d = vi < (n + VEC - 1) / VEC ? lds128(wb + kItemBytes + vi * 16) : neg_inf_vec(EB);
        unsigned long long wv[VEC];
        unsigned long long lsum = 0;
#pragma unroll
        for (int h = 0; h < VEC; ++h) {
          // past the end of the row (the unit's padding) the weight is 0
          const bool live = vi * VEC + h < n;
          wv[h] = live ? draw_weight<true>(vec_elem<EB>(t, h), vec_elem<EB>(d, h), kc) : 0ull;
          lsum += wv[h];
        }
        const unsigned long long li = warp_incl_scan_u64(lsum);
        unsigned long long r2 = run + li - lsum;
        int tk = -1;
        if (r2 <= target && target < r2 + lsum) {
#pragma unroll
          for (int h = 0; h < VEC; ++h) {
            if (tk < 0 && r2 + wv[h] > target) tk = unit_chunk(u) * AE + vi * VEC + h;
            r2 += wv[h];
          }
        }
        const unsigned int holder = __ballot_sync(0xffffffffu, tk >= 0);
        if (holder) tok = __shfl_sync(0xffffffffu, tk, __ffs(holder) - 1);
        else flags |= SV_STATUS_INTERNAL;
      }
      if (lane == 0) P.out_tokens[(size_t)b * (G + 1) + k] = tok;
      if (lane == 0) flags |= uflags;
    }
  }
  const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && any) atomicOr(P.status, any);
}

// Item j of a request in streaming order: its partial slot, chunk and row.
// Greedy steps stream target rows 0..gamma_b in order.  Sampled requests
// stream target row gamma_b (the bonus row) first, then the positions from
// the last down to 0, target row then draft row: the rows most often
// rejected (position 0) come last, closest to the residual pass that may
// re-read them.
struct StreamRow {
  int pslot, c, row;  // partial slot, chunk, row index within the target or draft rows
  bool draft;
};
__device__ __forceinline__ StreamRow stream_row(int j, int NC, int gb, bool greedy, int G) {
  StreamRow r;
  const int rr = j / NC;
  r.c = j - rr * NC;
  if (greedy || rr == 0) {
    r.row = greedy ? rr : gb;
    r.pslot = r.row;
    r.draft = false;
  } else {
    const int p = gb - 1 - (rr - 1) / 2;
    r.row = p;
    r.draft = ((rr - 1) & 1) != 0;
    r.pslot = r.draft ? G + 1 + p : p;
  }
  return r;
}

// ---------------------------------------------------------------------------
// Medium batches: one cluster per request, items streamed
// ---------------------------------------------------------------------------
// When a request's A work does not fit its cluster's warps one unit each, or
// only smaller clusters fit the batch in one wave, the warps of request b's
// cluster stream its items instead: warp gw of the cluster's W warps takes
// items gw, gw + W, gw + 2W, ... (item j is chunk j % NC of the request's row
// j / NC: target rows 0..gamma_b, then draft rows 0..gamma_b-1) through its
// staging buffers.  Partials go to every CTA's shared memory and a cluster barrier
// completes them, as on the resident path; every CTA's warp 0 computes the
// decision.  After a reject the warps stream row k's R chunks (target and
// draft halves, usually L2 hits) and store each chunk's fixed-point sum in
// the leader's shared memory; after a second barrier the leader's warp 0
// draws from those sums and walks one chunk.  With at most one request per
// cluster no global counter, record or queue is involved.  With more requests
// than clusters (clusters of one CTA) each CTA takes its requests one after
// another in a claim order (longest first, below): the first at its index,
// the next at a position from a global counter, claimed while the current one
// is decided; the other warps start the next request's items while warp 0
// draws.  Shared memory: the buffers, then (the same
// layout in every CTA) the partials [2G+1][NC] and the leader's chunk sums
// [NCR] (then, with claims, the claim order [B] and row counts [B]).  NW
// warps per CTA with NB staging buffers each; CPS CTAs per SM (two for greedy
// claims, so that one CTA's decision overlaps the other's streaming).  With
// one buffer per warp a sampling item moves into registers with its maximum
// and the buffer's next copy starts before the exponentials.
template <int EB, int MODE, bool PK, int NW, int NB, int CPS>
__global__ void __launch_bounds__(NW * 32, CPS) stream_kernel(Params P) {
  static_assert(NW * CPS * 32 <= 1024 && NB >= 1 && NB <= 2, "warps and buffers per SM");
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ __align__(8) uint64_t bar[NW][NB];
  __shared__ Meta smeta[NW][NB];  // the item in each buffer
  __shared__ float rsbuf[192];         // the decision's row statistics
  __shared__ ClusterDec sdec[2];  // by decision number: a warp reads one while the next is made
  __shared__ int s_next, s_last;       // the CTA's next claim; last CTA out
  __shared__ unsigned int s_ctr;       // tickets for the items of a phase
  __shared__ unsigned int s_dec;       // the latest decision: number << 1 | final
  __shared__ int s_hist[64];           // claim order: first position per row count
  __shared__ unsigned int s_rows;      // claims: the batch's rows
  constexpr int AE = kItemBytes / EB;   // logits per A item
  constexpr int RE = kHalfBytes / EB;   // logits per R chunk and row
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_size();
  const int nq = (int)(gridDim.x / C);  // clusters
  const bool queue = P.B > nq;          // requests claimed in turn (clusters of one CTA)
  const int G = P.G, V = P.V, NC = P.NC, NCR = P.NCR;
  float2* part = reinterpret_cast<float2*>(dsmem + (size_t)NW * NB * kItemBytes);
  unsigned long long* rsum = reinterpret_cast<unsigned long long*>(part + (size_t)(2 * G + 1) * NC);
  float2* bpart = reinterpret_cast<float2*>(rsum + NCR);  // the bonus row's partials, copied
  unsigned char* mybuf = dsmem + (size_t)warp * NB * kItemBytes;
  uint64_t* mybar = bar[warp];
  Meta* mymeta = smeta[warp];

  if (queue && C != 1) {  // claims are made for clusters of one CTA only
    if (tid == 0 && rank == 0) atomicOr(P.status, SV_STATUS_INTERNAL);
    return;
  }
  if (lane == 0) {
    for (int s = 0; s < NB; ++s) mbar_init(&mybar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid == 0) {
    s_ctr = 0;
    s_dec = ~0u;
  }
  __syncthreads();

  unsigned int issued = 0, processed = 0;  // copies started and consumed by this warp
  bool failed = false;
  unsigned int flags = 0;
  // Start the copy of item m into the next buffer (lane 0 issues it).
  auto issue = [&](const Meta& m) {
    const int s = (int)(issued % NB);
    if (lane == 0) {
      mymeta[s] = m;
      unsigned char* dst = mybuf + s * kItemBytes;
      if (m.direct) {
        mbar_arrive(&mybar[s]);
      } else {
        const unsigned int bytes = (unsigned int)(m.n * EB);
        const bool two = m.kind == KIND_R;
        mbar_arrive_expect_tx(&mybar[s], two ? 2 * bytes : bytes);
        bulk_copy_g2s(dst, m.p0, bytes, &mybar[s]);
        if (two) bulk_copy_g2s(dst + kHalfBytes, m.p1, bytes, &mybar[s]);
      }
    }
    __syncwarp();
    ++issued;
  };
  // Wait for the oldest copy in flight; false after the bounded wait gave up.
  auto wait_oldest = [&]() -> bool {
    if (mbar_wait(&mybar[processed % NB], (processed / NB) & 1u, P.wait_ns)) return true;
    flags |= SV_STATUS_TIMEOUT;
    failed = true;
    return false;
  };
  // Work within a phase (a stage's A items, or the R chunks) is taken from
  // a CTA counter: CTA r of the cluster takes the phase's items r, r + C,
  // r + 2C, ... in turn, so a warp that starts a phase late (warp 0 after a
  // draw) takes fewer.  Lane 0 requests the next ticket when it starts a
  // copy and reads it before the next one.  Every warp takes part in every
  // phase and stops at its first ticket past the phase's end, so a phase
  // uses n + NW tickets and every warp knows where the next one starts.
  // A cluster of one CTA meets at a CTA barrier: its stores through the
  // cluster window are to its own shared memory, and the CTA barrier is
  // cheaper than the cluster one (B = 512: 173.2 -> 170.5 us sampling,
  // 52.3 -> 50.8 us greedy).
  auto stage_sync = [&]() {
    if (C == 1) __syncthreads();
    else cluster_sync();
  };
  unsigned int tbase = 0, ticket = 0;
  unsigned int dseq = 0;  // decisions made by this CTA so far
  auto claim_next = [&]() {
    if (lane == 0) ticket = atomicAdd(&s_ctr, 1u);
  };
  auto claimed = [&]() -> unsigned int {  // index within this CTA's share
    return __shfl_sync(0xffffffffu, ticket, 0) - tbase;
  };
  auto share = [&](unsigned int n) -> unsigned int {  // this CTA's items of n
    return n > rank ? (n - rank + C - 1) / C : 0u;
  };

  // Claims are taken longest request first (by row count, then index): the
  // short requests claimed last fill in around the long ones.  Every CTA
  // builds the same order in shared memory: all threads read the row counts;
  // if they differ, warp 0 places each request with a stable counting sort
  // (about 3 us at B = 512, so a batch of equal counts keeps index order).
  int* order = reinterpret_cast<int*>(bpart + NC);                      // [B] requests by claim
  unsigned char* nrow = reinterpret_cast<unsigned char*>(order + P.B);  // [B] row counts
  bool sorted = false;  // claims go through `order`
  if (queue) {
    auto rows_of_req = [&](int b) -> int {
      int gb = 0;
      unsigned int fl = 0;
      if constexpr (PK) (void)packed_base(P, b, gb, fl);
      else gb = clamp_gamma(P.gamma ? P.gamma[b] : 0, G);
      const bool sampled = MODE == MODE_SAMPLE && P.temperature[b] != 0.0f;
      return sampled ? 2 * gb + 1 : gb + 1;
    };
    const int r0 = rows_of_req(0);
    int differs = 0;
    unsigned int rows = 0;
    if (tid == 0) s_rows = 0;
    __syncthreads();
#pragma unroll 4
    for (int b = tid; b < P.B; b += NW * 32) {
      const int r = rows_of_req(b);
      nrow[b] = (unsigned char)r;
      differs |= r != r0;
      rows += (unsigned int)r;
    }
    rows = __reduce_add_sync(0xffffffffu, rows);
    if (lane == 0) atomicAdd(&s_rows, rows);
    sorted = __syncthreads_or(differs) != 0;
  }
  if (sorted) {
    if (warp == 0) {
      for (int r = lane; r < 64; r += 32) s_hist[r] = 0;
      __syncwarp();
      // counts per row count: one add per distinct count in each group of 32
      for (int b0 = 0; b0 < P.B; b0 += 32) {
        const int b = b0 + lane;
        const int r = b < P.B ? (int)nrow[b] : 64;  // 64: past the batch
        const unsigned int peers = __match_any_sync(0xffffffffu, r);
        if (r < 64 && lane == __ffs(peers) - 1) s_hist[r] += __popc(peers);
        __syncwarp();
      }
      // first position of each row count, longest first: lane l holds counts
      // 2l and 2l + 1; a suffix sum over the lanes
      const int h0 = s_hist[2 * lane], h1 = s_hist[2 * lane + 1];
      int suf = h0 + h1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      const int after = suf - h0 - h1;  // requests with more rows than 2l + 1
      __syncwarp();
      s_hist[2 * lane + 1] = after;
      s_hist[2 * lane] = after + h1;
      __syncwarp();
      for (int b0 = 0; b0 < P.B; b0 += 32) {
        const int b = b0 + lane;
        const int r = b < P.B ? (int)nrow[b] : 64;  // 64: past the batch
        const unsigned int peers = __match_any_sync(0xffffffffu, r);
        const int before = __popc(peers & ((1u << lane) - 1u));
        if (r < 64) order[s_hist[r] + before] = b;
        __syncwarp();
        if (r < 64 && before == 0) s_hist[r] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
  }

  for (int claim = (int)cluster_index(); claim < P.B;) {
    const int b = sorted ? order[claim] : claim;
    // the request: draft length, addresses, temperature constants
    unsigned int rflags = 0;
    int gb = 0, base = 0;
    if constexpr (PK) {
      base = packed_base(P, b, gb, rflags);
    } else {
      const int g_in = P.gamma ? P.gamma[b] : 0;
      gb = clamp_gamma(g_in, G);
      if (g_in != gb) rflags |= SV_STATUS_BAD_GAMMA;
    }
    const ReqAddr A = addr_from_base<PK>(P, b, base, gb);
    bool greedy = MODE == MODE_GREEDY;
    TempC tc{0.0f, 0.0f};
    if (MODE == MODE_SAMPLE) {
      const float T = P.temperature[b];
      if (T == 0.0f) greedy = true;  // this request takes the greedy steps
      else tc = temp_consts(sanitize_temperature(T, rflags));
    }
    const bool sample = MODE == MODE_SAMPLE && !greedy;
    // every CTA decides: its warp 0 requests the draft inputs and the final
    // draw's uniform before its items
    DraftIn gin{0, 0.0f, 0.0f, 0.0f, 0u};
    float u_fin = 0.0f;
    unsigned int uflags = 0;
    if (sample && warp == 0) {
      gin = gather_drafts<EB>(P, A, gb);
      u_fin = sanitize_uniform(P.uniforms[A.uf], uflags);
    }

    // The A items come in stages, each followed by the decision over its
    // positions.  With claims a sampled request is taken lazily: stage s
    // holds target and draft rows s only, and the rows of position s + 1
    // matter only if draft s is accepted (the stage after the last position
    // holds the bonus row gamma_b).  For a request with at least
    // kSpecMinGamma drafts the other warps already stream stage s + 1 while
    // warp 0 decides stage s; if the decision is final they stop taking its
    // items, and what they read of it is not used.  Otherwise one stage holds
    // every row.  Each position's arithmetic is the same either way.
    // Lazy stages lengthen a request while they shorten the batch's work, so
    // sampled requests are read this way where requests queue at least two
    // deep per CTA, and not when a request's rows alone reach 80 % of a CTA's
    // average share of the batch (the call lasts at least as long as that
    // request does).  Measured: B = 512, gamma 1 and 3: 112 -> 110 and 201 ->
    // 170 us; B = 256 ragged (1.7 requests per CTA): 131 eager against 135
    // lazy.  Greedy steps read one target row per stage, and no residual pass
    // follows a mismatch: B = 512, gamma 3: 80 -> 50 us.
    const bool lazy = P.lazy && queue &&
                      (!sample || (P.B >= 2 * nq &&
                                   5ull * (unsigned long long)(2 * gb + 1) * (unsigned long long)nq <
                                       4ull * (unsigned long long)s_rows));
    // a stage's end: sampled, positions [slo, hi) (plus the bonus row when
    // slo == gamma_b, or eagerly); greedy, target rows [slo, hi)
    auto stage_hi = [&](int slo) {
      return sample ? (lazy ? min(slo + 1, gb) : gb) : (lazy ? slo + 1 : gb + 1);
    };
    // The items of the stage that starts at position slo.  With `spec` the
    // warp stops taking them once the decision in progress (number dseq) is
    // final; it still draws its remaining tickets, so that the stage uses
    // its usual count.
    auto run_stage = [&](int slo, bool spec) {
      const int hi = stage_hi(slo);
      const bool with_bonus = !lazy || slo == gb;
      const int npos = hi - slo;
      const int nrows = !sample ? npos : 2 * npos + (with_bonus ? 1 : 0);
      const unsigned int nI = (unsigned int)nrows * (unsigned int)NC;
      auto a_meta = [&](unsigned int j) {
        // the rows in streaming order: eagerly, a sampled request's position-0
        // rows, the most often rejected, come last, closest to the residual
        // pass; lazily, target row slo then draft row slo (or the bonus row)
        StreamRow fr;
        if (lazy && sample) {
          const int rr = (int)j / NC;
          fr.c = (int)j - rr * NC;
          fr.draft = rr == 1;
          fr.row = npos ? slo : gb;
          fr.pslot = fr.draft ? G + 1 + slo : fr.row;
        } else if (lazy) {  // greedy: target row slo
          fr.c = (int)j;
          fr.draft = false;
          fr.row = slo;
          fr.pslot = slo;
        } else {
          fr = stream_row((int)j, NC, gb, !sample, G);
        }
        const int c = fr.c;
        Meta m;
        const size_t roff = ((fr.draft ? A.d0 : A.t0) + (size_t)fr.row) * (size_t)V;
        const char* rows = fr.draft ? P.draft : P.target;
        m.pslot = fr.pslot;
        m.kind = KIND_A;
        m.b = b;
        m.c = c;
        m.n = min(AE, V - c * AE);
        m.reject = 0;
        m.pad = 0;
        m.p0 = rows + (roff + (size_t)c * AE) * EB;
        m.p1 = nullptr;
        m.direct = ((reinterpret_cast<uintptr_t>(m.p0) & 15) != 0 || ((m.n * EB) & 15) != 0) ? 1 : 0;
        m.mt = m.md = m.inv_st = m.rho = 0.0f;
        m.c_hi = tc.hi;
        m.c_lo = tc.lo;
        return m;
      };
      // lane r < C stores each partial into CTA r: every CTA decides locally
      const uint32_t part_r = rank_addr(part, (uint32_t)lane < C ? (uint32_t)lane : 0u);
      auto store_at = [&](int pslot, int c, float2 pr) {
        if ((uint32_t)lane < C)
          st_cluster_f2(part_r + (uint32_t)((pslot * NC + c) * (int)sizeof(float2)), pr);
      };
      auto store_part = [&](const Meta& m, float2 pr) { store_at(m.pslot, m.c, pr); };
      const unsigned int nA = share(nI);
      const unsigned int final_tag = (dseq << 1) | 1u;
      bool more = true;  // this warp's tickets have not yet run past the stage
      bool dropped = false;
      claim_next();
      auto top_up = [&]() {  // start copies into every free buffer
        while (more && !dropped && issued - processed < (unsigned int)NB) {
          if (spec && *reinterpret_cast<volatile unsigned int*>(&s_dec) == final_tag) {
            dropped = true;
            break;
          }
          const unsigned int t = claimed();
          if (t >= nA) {
            more = false;
          } else {
            issue(a_meta(rank + C * t));
            claim_next();
          }
        }
      };
      while (!failed) {
        top_up();
        if (issued == processed || !wait_oldest()) break;
        const Meta& m = mymeta[processed % NB];
        char* stage = reinterpret_cast<char*>(mybuf + (processed % NB) * kItemBytes);
        const bool padded = !m.direct && m.n < AE;  // a row's last chunk
        const bool written = (sample && m.direct) || padded;
        if (sample && m.direct) stage_unaligned<EB>(m, stage);
        else if (padded) pad_item_tail<EB>(stage, m.n);
        const int pslot = m.pslot, c = m.c;
        if (NB == 1 && sample) {
          // the item moves into registers with its maximum; the buffer's next
          // copy then runs during the exponentials
          const float c_hi = m.c_hi, c_lo = m.c_lo;
          uint32_t w[kItemWords];
          const float mx = item_load_max<EB>(stage, w);
          // stores into the buffer are ordered before the next bulk copy into it
          if (written) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          ++processed;
          top_up();
          store_at(pslot, c, make_float2(mx, item_exp_sum<EB>(w, mx, c_hi, c_lo)));
        } else {
          store_at(pslot, c, sample ? a_item_sample<EB>(m, stage) : a_item_greedy<EB>(m, stage));
          if (written) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          ++processed;
        }
      }
      if (failed) {
        // Every item of this warp still stores a partial, (NaN, 0) where it
        // could not be read: every CTA then holds the same table and takes the
        // same branches below.  Copies in flight are waited for (bounded).
        for (; processed != issued; ++processed) {
          (void)mbar_wait(&mybar[processed % NB], (processed / NB) & 1u, P.wait_ns);
          store_part(mymeta[processed % NB], make_float2(NAN, 0.0f));
          __syncwarp();
        }
      }
      // tickets left after a failure or a dropped stage
      while (more) {
        const unsigned int t = claimed();
        if (t >= nA) {
          more = false;
        } else {
          if (!dropped) store_part(a_meta(rank + C * t), make_float2(NAN, 0.0f));
          claim_next();
        }
      }
      tbase += nA + NW;
    };

    ClusterDec cd;
    run_stage(0, false);
    stage_sync();  // every CTA holds every partial of the first stage
    // greedy: no further cluster work (with claims, C == 1: every CTA leads)
    if (greedy && rank != 0) return;
    for (int lo = 0;;) {
      const int hi = stage_hi(lo);
      const bool with_bonus = !lazy || lo == gb;
      // ---- the decision (as on the resident cluster path)
      if (warp == 0) {
        // queue: the next request is claimed now, its latency hidden by the decision
        unsigned int nclaim = 0;
        if (lane == 0 && lo == 0 && queue) nclaim = atomicAdd(P.next_item, 1u);
        float* rs = rsbuf;
        const SharedParts sp{part, NC};
        ClusterDec dc;
        dc.k = 0;
        dc.go = 0;
        dc.mt = dc.md = dc.inv_st = dc.rho = 0.0f;
        dc.c_hi = tc.hi;
        dc.c_lo = tc.lo;
        if (greedy) {
          dc.k = greedy_range<PK>(P, sp, b, gb, reinterpret_cast<int*>(rs), lo, hi);
        } else {
          Decision d;
          d.k = 0;
          d.reject = 0;
          d.mt = d.md = d.inv_st = d.rho = 0.0f;
          const int k = decide_range<EB, PK>(P, sp, b, gb, tc, rs, A, gin, d, lo, hi,
                                             with_bonus, rank == 0);
          dc.k = k;
          dc.go = __shfl_sync(0xffffffffu, d.reject, 0);
          dc.mt = __shfl_sync(0xffffffffu, d.mt, 0);
          dc.md = __shfl_sync(0xffffffffu, d.md, 0);
          dc.inv_st = __shfl_sync(0xffffffffu, d.inv_st, 0);
          dc.rho = __shfl_sync(0xffffffffu, d.rho, 0);
          // every draft accepted: the leader draws the bonus token after the
          // CTA's other warps have moved on, from a copy of the row's partials
          // (the next request's items overwrite the table)
          if (k == gb && rank == 0) {
            for (int c = lane; c < NC; c += 32) bpart[c] = part[gb * NC + c];
            __syncwarp();
          }
        }
        if (lane == 0) {
          if (lo == 0) s_next = queue ? (int)nclaim + nq : P.B;
          sdec[dseq & 1] = dc;
          if (dc.k >= 0 && rank == 0 && rflags) atomicOr(P.status, rflags);
          *reinterpret_cast<volatile unsigned int*>(&s_dec) = (dseq << 1) | (dc.k >= 0 ? 1u : 0u);
        }
        __syncwarp();
      }
      // the next stage, read while the decision is made, or once it is known
      const bool spec = lazy && sample && hi < gb && gb >= kSpecMinGamma;
      if (spec) run_stage(hi, true);
      __syncthreads();  // the CTA's warps see the decision
      cd = sdec[dseq & 1];
      ++dseq;
      if (cd.k >= 0) break;
      if (!spec) {
        run_stage(hi, false);
        stage_sync();  // every partial of the stage
      }
      lo = hi;  // every draft of the stage accepted: its next stage is in
    }  // stages
    const int next = s_next;
    if (sample && cd.k == gb && rank == 0 && warp == 0)  // its copies are all consumed
      final_bonus<EB, PK>(P, RowParts{bpart}, b, gb, tc, cd.mt, mybuf);

    if (cd.go) {
      // ---- the residual chunk sums of the rejected position k (k < gamma_b)
      const int k = cd.k < 0 ? 0 : (cd.k > G ? G : cd.k);
      const char* trow = P.target + (A.t0 + (size_t)k) * (size_t)V * EB;
      const char* drow = P.draft + (A.d0 + (size_t)k) * (size_t)V * EB;
      auto r_meta = [&](unsigned int c) {
        Meta m;
        m.kind = KIND_R;
        m.b = b;
        m.pslot = k;
        m.c = (int)c;
        m.n = min(RE, V - (int)c * RE);
        m.reject = 1;
        m.pad = 0;
        m.p0 = trow + (size_t)c * RE * EB;
        m.p1 = drow + (size_t)c * RE * EB;
        const uintptr_t a = reinterpret_cast<uintptr_t>(m.p0) | reinterpret_cast<uintptr_t>(m.p1);
        m.direct = ((a & 15) != 0 || ((m.n * EB) & 15) != 0) ? 1 : 0;
        m.mt = cd.mt;
        m.md = cd.md;
        m.inv_st = cd.inv_st;
        m.rho = cd.rho;
        m.c_hi = cd.c_hi;
        m.c_lo = cd.c_lo;
        return m;
      };
      const uint32_t rsum0 = rank_addr(rsum, 0u);  // the leader's chunk sums
      const unsigned int nR = share((unsigned int)NCR);
      bool more = true;
      claim_next();
      while (!failed) {
        while (more && issued - processed < (unsigned int)NB) {
          const unsigned int t = claimed();
          if (t >= nR) {
            more = false;
          } else {
            issue(r_meta(rank + C * t));
            claim_next();
          }
        }
        if (issued == processed || !wait_oldest()) break;
        const Meta& m = mymeta[processed % NB];
        const unsigned long long sr =
            r_item<EB>(m, reinterpret_cast<const char*>(mybuf + (processed % NB) * kItemBytes));
        if (lane == 0) st_cluster_u64(rsum0 + (uint32_t)m.c * 8u, sr);
        __syncwarp();
        ++processed;
      }
      if (failed) {  // copies in flight are waited for (bounded); missing sums are 0
        for (; processed != issued; ++processed) {
          (void)mbar_wait(&mybar[processed % NB], (processed / NB) & 1u, P.wait_ns);
          if (lane == 0) st_cluster_u64(rsum0 + (uint32_t)mymeta[processed % NB].c * 8u, 0ull);
          __syncwarp();
        }
        while (more) {
          const unsigned int t = claimed();
          if (t >= nR) {
            more = false;
          } else {
            if (lane == 0) st_cluster_u64(rsum0 + (rank + C * t) * 8u, 0ull);
            __syncwarp();
            claim_next();
          }
        }
      }
      tbase += nR + NW;
      stage_sync();  // the leader holds every chunk sum

      // ---- the final draw: the leader's warp 0 (its copies are all consumed)
      if (rank == 0 && warp == 0) {
        ResidC kc;
        kc.mt = cd.mt; kc.md = cd.md; kc.inv_st = cd.inv_st; kc.rho = cd.rho;
        resid_scales(kc);
        kc.hi = cd.c_hi; kc.lo = cd.c_lo; kc.reject = 1;
        int tok = chunk_draw<EB, false>(trow, drow, V, NCR, u_fin, kc, rsum, mybuf);
        if (lane == 0) {
          if (tok < 0) {
            flags |= SV_STATUS_INTERNAL;
            tok = V - 1;
          }
          P.out_tokens[(size_t)b * (G + 1) + k] = tok;
          flags |= uflags;
        }
      }
    }
    claim = next;
  }  // requests
  const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && any) atomicOr(P.status, any);
  if (queue) {
    // the last CTA out resets the claim counter for the next call
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      s_last = atomicAdd(P.exit_count, 1u) == gridDim.x - 1 ? 1 : 0;
    }
    __syncthreads();
    if (s_last && tid == 0) {
      *P.next_item = 0;
      *P.exit_count = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Request claims as a pipeline: two requests in flight per CTA
// ---------------------------------------------------------------------------
// The streaming kernel's claims take a request's stages one after another,
// each ending in a CTA barrier and a decision that one warp computes while
// the others wait.  Here a CTA keeps two requests (slots) in flight and its
// work as a list of phases: a stage of one slot's request (its A items) or
// its residual pass (R items).  Warps take the items of the oldest phase with
// items left, so when one phase runs out they move on to the other slot's
// without a barrier.  The warp that completes a phase's last item runs what
// follows: the decision (the next stage, the residual pass, or the bonus
// draw), the final draw, and the claim and set-up of the slot's next request,
// each appending that slot's next phase.  A slot's phases follow one another
// in order, so each request's arithmetic is that of the streaming kernel.
// Every wait is bounded; the last CTA out resets the claim counter.
constexpr int kPipeSlots = 2;
constexpr int kPipeRing = 16;  // phase records, reused in turn
constexpr int kPipeWarps = 16;

struct PipePhase {
  int seq;           // sequence number of the phase this record holds
  int slot;
  int kind;          // KIND_A: a stage; KIND_R: the residual pass
  int lo, hi;        // A: positions [lo, hi) (sampled) or target rows [lo, hi) (greedy)
  int bonus;         // A, sampled: the bonus row is in the stage
  unsigned int n;    // items
  unsigned int tickets;
  unsigned int done;
};
struct PipeSlot {
  int b, gb, sample, lazy;
  ReqAddr A;
  TempC tc;
  unsigned int rflags, uflags;
  float u_fin;
  int x[32];
  float u[32], zt[32], zd[32];
  unsigned int gfl[32];
  Decision d;        // the rejection's decision, for the residual pass and draw
  float rs[192];     // row statistics (sampled) or argmax per row (greedy)
};

template <int EB, bool PK, int NW>
__global__ void __launch_bounds__(NW * 32, 1) pipe_kernel(Params P) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ __align__(8) uint64_t bar[NW];
  __shared__ Meta smeta[NW];
  __shared__ PipePhase ring[kPipeRing];
  __shared__ PipeSlot slots[kPipeSlots];
  __shared__ unsigned int s_pub;      // phases published (in order)
  __shared__ unsigned int s_alloc;    // phases reserved
  __shared__ int s_live;              // slots with a request
  __shared__ int s_pseq[NW];          // the oldest phase each warp may still read (ring reuse)
  __shared__ int s_last;
  __shared__ unsigned int s_rows;
  __shared__ int s_hist[64];
  constexpr int AE = kItemBytes / EB;
  constexpr int RE = kHalfBytes / EB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G, V = P.V, NC = P.NC, NCR = P.NCR;
  const int nq = (int)gridDim.x;
  // dynamic shared memory: buffers | per slot: partials, chunk sums, draw stage | order | rows
  const size_t part_b = (((size_t)(2 * G + 1) * NC * sizeof(float2)) + 15) & ~(size_t)15;
  const size_t rsum_b = (((size_t)NCR * sizeof(unsigned long long)) + 15) & ~(size_t)15;
  const size_t slot_b = part_b + rsum_b + kItemBytes;
  unsigned char* slot_base = dsmem + (size_t)NW * kItemBytes;
  auto s_part = [&](int sl) { return reinterpret_cast<float2*>(slot_base + sl * slot_b); };
  auto s_rsum = [&](int sl) {
    return reinterpret_cast<unsigned long long*>(slot_base + sl * slot_b + part_b);
  };
  auto s_stage = [&](int sl) { return slot_base + sl * slot_b + part_b + rsum_b; };
  int* order = reinterpret_cast<int*>(slot_base + kPipeSlots * slot_b);
  unsigned char* nrow = reinterpret_cast<unsigned char*>(order + P.B);
  unsigned char* mybuf = dsmem + (size_t)warp * kItemBytes;
  unsigned int flags = 0;

  if (lane == 0) {
    mbar_init(&bar[warp], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid == 0) {
    s_pub = 0;
    s_alloc = 0;
    s_live = kPipeSlots;
    s_rows = 0;
  }
  if (tid < kPipeRing) ring[tid].seq = -1;
  if (lane == 0) s_pseq[warp] = 0;
  __syncthreads();

  // the claim order, longest first (as the streaming kernel builds it)
  auto rows_of_req = [&](int b) -> int {
    int gb = 0;
    unsigned int fl = 0;
    if constexpr (PK) (void)packed_base(P, b, gb, fl);
    else gb = clamp_gamma(P.gamma ? P.gamma[b] : 0, G);
    return P.temperature[b] != 0.0f ? 2 * gb + 1 : gb + 1;
  };
  bool sorted = false;
  {
    const int r0 = rows_of_req(0);
    int differs = 0;
    unsigned int rows = 0;
    for (int b = tid; b < P.B; b += NW * 32) {
      const int r = rows_of_req(b);
      nrow[b] = (unsigned char)r;
      differs |= r != r0;
      rows += (unsigned int)r;
    }
    rows = __reduce_add_sync(0xffffffffu, rows);
    if (lane == 0) atomicAdd(&s_rows, rows);
    sorted = __syncthreads_or(differs) != 0;
  }
  if (sorted) {
    if (warp == 0) {
      for (int r = lane; r < 64; r += 32) s_hist[r] = 0;
      __syncwarp();
      for (int b0 = 0; b0 < P.B; b0 += 32) {
        const int b = b0 + lane;
        const int r = b < P.B ? (int)nrow[b] : 64;
        const unsigned int peers = __match_any_sync(0xffffffffu, r);
        if (r < 64 && lane == __ffs(peers) - 1) s_hist[r] += __popc(peers);
        __syncwarp();
      }
      const int h0 = s_hist[2 * lane], h1 = s_hist[2 * lane + 1];
      int suf = h0 + h1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      const int after = suf - h0 - h1;
      __syncwarp();
      s_hist[2 * lane + 1] = after;
      s_hist[2 * lane] = after + h1;
      __syncwarp();
      for (int b0 = 0; b0 < P.B; b0 += 32) {
        const int b = b0 + lane;
        const int r = b < P.B ? (int)nrow[b] : 64;
        const unsigned int peers = __match_any_sync(0xffffffffu, r);
        const int before = __popc(peers & ((1u << lane) - 1u));
        if (r < 64) order[s_hist[r] + before] = b;
        __syncwarp();
        if (r < 64 && before == 0) s_hist[r] += __popc(peers);
        __syncwarp();
      }
    }
    __syncthreads();
  }

  // ---- phases (one warp at a time appends; lane 0 writes)
  // a stage's end: sampled, positions [lo, hi); greedy, target rows [lo, hi)
  auto stage_hi = [&](const PipeSlot& S, int lo) {
    return S.sample ? (S.lazy ? min(lo + 1, S.gb) : S.gb) : (S.lazy ? lo + 1 : S.gb + 1);
  };
  auto append = [&](int sl, int kind, int lo) {
    PipeSlot& S = slots[sl];
    int hi = 0, bonus = 0;
    unsigned int n;
    if (kind == KIND_A) {
      hi = stage_hi(S, lo);
      bonus = S.sample && (!S.lazy || lo == S.gb);
      const int npos = hi - lo;
      const int nrows = S.sample ? 2 * npos + bonus : npos;
      n = (unsigned int)nrows * (unsigned int)NC;
    } else {
      n = (unsigned int)NCR;
    }
    if (lane == 0) {
      const unsigned int seq = atomicAdd(&s_alloc, 1u);  // two slots may append at once
      // the record is reused once every warp has moved past its last use
      const unsigned long long t0 = now_ns();
      for (;;) {
        int lag = 0;
        for (int w = 0; w < NW; ++w)
          lag |= (int)seq - *reinterpret_cast<volatile int*>(&s_pseq[w]) >= kPipeRing;
        if (!lag) break;
        if (now_ns() - t0 > P.wait_ns) {
          flags |= SV_STATUS_TIMEOUT;
          break;
        }
        __nanosleep(64);
      }
      PipePhase& r = ring[seq % kPipeRing];
      r.slot = sl;
      r.kind = kind;
      r.lo = lo;
      r.hi = hi;
      r.bonus = bonus;
      r.n = n;
      r.tickets = 0;
      r.done = 0;
      r.seq = (int)seq;
      __threadfence_block();
      // published in order: after every earlier phase
      const unsigned long long t1 = now_ns();
      while (*reinterpret_cast<volatile unsigned int*>(&s_pub) != seq && now_ns() - t1 <= P.wait_ns)
        __nanosleep(32);
      if (*reinterpret_cast<volatile unsigned int*>(&s_pub) == seq)
        *reinterpret_cast<volatile unsigned int*>(&s_pub) = seq + 1;
      else
        flags |= SV_STATUS_TIMEOUT;
    }
    __syncwarp();
  };

  // ---- a slot's request: claim c of the order (or retire the slot)
  auto start = [&](int sl, int claim) {
    PipeSlot& S = slots[sl];
    if (claim >= P.B) {
      if (lane == 0) atomicSub(&s_live, 1);
      __syncwarp();
      return;
    }
    const int b = sorted ? order[claim] : claim;
    unsigned int rflags = 0;
    int gb = 0, base = 0;
    if constexpr (PK) {
      base = packed_base(P, b, gb, rflags);
    } else {
      const int g_in = P.gamma ? P.gamma[b] : 0;
      gb = clamp_gamma(g_in, G);
      if (g_in != gb) rflags |= SV_STATUS_BAD_GAMMA;
    }
    const ReqAddr A = addr_from_base<PK>(P, b, base, gb);
    TempC tc{0.0f, 0.0f};
    const float T = P.temperature[b];
    const bool sample = T != 0.0f;
    if (sample) tc = temp_consts(sanitize_temperature(T, rflags));
    const bool lazy = P.lazy && P.B >= 2 * nq &&
                      (!sample || 5ull * (unsigned long long)(2 * gb + 1) * (unsigned long long)nq <
                                      4ull * (unsigned long long)s_rows);
    DraftIn g{0, 0.0f, 0.0f, 0.0f, 0u};
    unsigned int uflags = 0;
    float u_fin = 0.0f;
    if (sample) {
      g = gather_drafts<EB>(P, A, gb);
      u_fin = sanitize_uniform(P.uniforms[A.uf], uflags);
    }
    S.x[lane] = g.x;
    S.u[lane] = g.u;
    S.zt[lane] = g.zt;
    S.zd[lane] = g.zd;
    S.gfl[lane] = g.flags;
    if (lane == 0) {
      S.b = b;
      S.gb = gb;
      S.sample = sample ? 1 : 0;
      S.lazy = lazy ? 1 : 0;
      S.A = A;
      S.tc = tc;
      S.rflags = rflags;
      S.uflags = uflags;
      S.u_fin = u_fin;
    }
    __syncwarp();
    append(sl, KIND_A, 0);
  };
  auto finish = [&](int sl) {
    int c = 0;
    if (lane == 0) c = (int)atomicAdd(P.next_item, 1u) + nq;
    c = __shfl_sync(0xffffffffu, c, 0);
    start(sl, c);
  };

  // ---- what follows a phase's last item (one warp)
  auto follow = [&](const PipePhase& ph) {
    const int sl = ph.slot;
    PipeSlot& S = slots[sl];
    const SharedParts sp{s_part(sl), NC};
    if (ph.kind == KIND_A) {
      int k;
      if (!S.sample) {
        k = greedy_range<PK>(P, sp, S.b, S.gb, reinterpret_cast<int*>(S.rs), ph.lo, ph.hi);
      } else {
        DraftIn g;
        g.x = S.x[lane];
        g.u = S.u[lane];
        g.zt = S.zt[lane];
        g.zd = S.zd[lane];
        g.flags = S.gfl[lane];
        Decision d;
        d.k = 0;
        d.reject = 0;
        d.mt = d.md = d.inv_st = d.rho = 0.0f;
        k = decide_range<EB, PK>(P, sp, S.b, S.gb, S.tc, S.rs, S.A, g, d, ph.lo, ph.hi, ph.bonus != 0,
                                 true);
        if (k >= 0 && lane == 0) S.d = d;
        __syncwarp();
      }
      if (k < 0) {
        append(sl, KIND_A, ph.hi);
        return;
      }
      if (lane == 0 && S.rflags) atomicOr(P.status, S.rflags);
      if (S.sample && k < S.gb) {
        append(sl, KIND_R, k);
        return;
      }
      if (S.sample)  // every draft accepted: the bonus token
        final_bonus<EB, PK>(P, sp, S.b, S.gb, S.tc, S.rs[S.gb], s_stage(sl));
      finish(sl);
      return;
    }
    // the residual pass is complete: the draw
    const int k = S.d.k < 0 ? 0 : (S.d.k > G ? G : S.d.k);
    const char* trow = P.target + (S.A.t0 + (size_t)k) * (size_t)V * EB;
    const char* drow = P.draft + (S.A.d0 + (size_t)k) * (size_t)V * EB;
    ResidC kc;
    kc.mt = S.d.mt; kc.md = S.d.md; kc.inv_st = S.d.inv_st; kc.rho = S.d.rho;
    resid_scales(kc);
    kc.hi = S.tc.hi; kc.lo = S.tc.lo; kc.reject = 1;
    int tok = chunk_draw<EB, false>(trow, drow, V, NCR, S.u_fin, kc, s_rsum(sl), s_stage(sl));
    if (lane == 0) {
      if (tok < 0) {
        flags |= SV_STATUS_INTERNAL;
        tok = V - 1;
      }
      P.out_tokens[(size_t)S.b * (G + 1) + k] = tok;
      flags |= S.uflags;
    }
    __syncwarp();
    finish(sl);
  };

  // ---- the item of ticket t of phase seq
  auto make_meta = [&](int seq, unsigned int t) {
    const PipePhase& ph = ring[seq % kPipeRing];
    const PipeSlot& S = slots[ph.slot];
    Meta m;
    m.pad = seq;
    m.b = S.b;
    m.c_hi = S.tc.hi;
    m.c_lo = S.tc.lo;
    if (ph.kind == KIND_A) {
      StreamRow fr;
      if (S.lazy && S.sample) {
        const int rr = (int)t / NC;
        fr.c = (int)t - rr * NC;
        fr.draft = rr == 1;
        fr.row = ph.hi > ph.lo ? ph.lo : S.gb;
        fr.pslot = fr.draft ? G + 1 + ph.lo : fr.row;
      } else if (S.lazy) {
        fr.c = (int)t;
        fr.draft = false;
        fr.row = ph.lo;
        fr.pslot = ph.lo;
      } else {
        fr = stream_row((int)t, NC, S.gb, !S.sample, G);
      }
      const size_t roff = ((fr.draft ? S.A.d0 : S.A.t0) + (size_t)fr.row) * (size_t)V;
      m.kind = KIND_A;
      m.pslot = fr.pslot;
      m.c = fr.c;
      m.n = min(AE, V - fr.c * AE);
      m.reject = 0;
      m.p0 = (fr.draft ? P.draft : P.target) + (roff + (size_t)fr.c * AE) * EB;
      m.p1 = nullptr;
      m.direct = ((reinterpret_cast<uintptr_t>(m.p0) & 15) != 0 || ((m.n * EB) & 15) != 0) ? 1 : 0;
      m.mt = m.md = m.inv_st = m.rho = 0.0f;
    } else {
      const int k = S.d.k < 0 ? 0 : (S.d.k > G ? G : S.d.k);
      m.kind = KIND_R;
      m.pslot = k;
      m.c = (int)t;
      m.n = min(RE, V - (int)t * RE);
      m.reject = 1;
      m.p0 = P.target + ((S.A.t0 + (size_t)k) * (size_t)V + (size_t)t * RE) * EB;
      m.p1 = P.draft + ((S.A.d0 + (size_t)k) * (size_t)V + (size_t)t * RE) * EB;
      const uintptr_t a = reinterpret_cast<uintptr_t>(m.p0) | reinterpret_cast<uintptr_t>(m.p1);
      m.direct = ((a & 15) != 0 || ((m.n * EB) & 15) != 0) ? 1 : 0;
      m.mt = S.d.mt;
      m.md = S.d.md;
      m.inv_st = S.d.inv_st;
      m.rho = S.d.rho;
    }
    return m;
  };

  // ---- the first two requests: this CTA's index and one claim
  if (warp == 0) {
    start(0, (int)blockIdx.x);
  } else if (warp == 1) {
    int c = 0;
    if (lane == 0) c = (int)atomicAdd(P.next_item, 1u) + nq;
    c = __shfl_sync(0xffffffffu, c, 0);
    start(1, c);
  }
  __syncthreads();

  // ---- the warps' loop
  unsigned int issued = 0, processed = 0;
  int pseq = 0;          // the phase this warp takes tickets from
  int hold = INT_MAX;    // the phase of the item this warp is processing
  int shown = 0;         // what s_pseq[warp] holds
  bool failed = false;
  // a ticket of the oldest phase with tickets left: 1 (seq, t), 0 none yet, -1 all done
  auto claim = [&](int& seq, unsigned int& t) -> int {
    for (;;) {
      const unsigned int pub = *reinterpret_cast<volatile unsigned int*>(&s_pub);
      if ((unsigned int)pseq >= pub) {
        return *reinterpret_cast<volatile int*>(&s_live) == 0 ? -1 : 0;
      }
      unsigned int got = 0;
      if (lane == 0) got = atomicAdd(&ring[pseq % kPipeRing].tickets, 1u);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (got < ring[pseq % kPipeRing].n) {
        seq = pseq;
        t = got;
        return 1;
      }
      ++pseq;
      if (min(pseq, hold) != shown) {
        shown = min(pseq, hold);
        if (lane == 0) *reinterpret_cast<volatile int*>(&s_pseq[warp]) = shown;
      }
    }
  };
  auto issue = [&](int seq, unsigned int t) {
    const Meta m = make_meta(seq, t);
    if (lane == 0) {
      smeta[warp] = m;
      if (m.direct) {
        mbar_arrive(&bar[warp]);
      } else {
        const unsigned int bytes = (unsigned int)(m.n * EB);
        const bool two = m.kind == KIND_R;
        mbar_arrive_expect_tx(&bar[warp], two ? 2 * bytes : bytes);
        bulk_copy_g2s(mybuf, m.p0, bytes, &bar[warp]);
        if (two) bulk_copy_g2s(mybuf + kHalfBytes, m.p1, bytes, &bar[warp]);
      }
    }
    __syncwarp();
    ++issued;
  };
  auto top_up = [&]() -> int {  // a copy in flight: 1; none and none to come: -1
    if (issued != processed) return 1;
    int seq;
    unsigned int t;
    const int r = claim(seq, t);
    if (r == 1) issue(seq, t);
    return r;
  };
  const unsigned long long idle_limit = P.wait_ns;
  while (!failed) {
    int r = top_up();
    if (r < 0) break;
    if (r == 0) {  // nothing published yet: wait (bounded)
      const unsigned long long t0 = now_ns();
      while ((r = top_up()) == 0 && now_ns() - t0 <= idle_limit) __nanosleep(128);
      if (r < 0) break;
      if (r == 0) {
        flags |= SV_STATUS_TIMEOUT;
        break;
      }
    }
    if (!mbar_wait(&bar[warp], processed & 1u, P.wait_ns)) {
      flags |= SV_STATUS_TIMEOUT;
      failed = true;
      break;
    }
    const Meta& m = smeta[warp];
    const int seq = m.pad;
    hold = seq;  // kept until the item is counted (the record stays while the warp reads it)
    const int sl = ring[seq % kPipeRing].slot;
    char* stage = reinterpret_cast<char*>(mybuf);
    if (m.kind == KIND_A) {
      const bool smp = slots[sl].sample != 0;
      const bool padded = !m.direct && m.n < AE;
      const bool written = (smp && m.direct) || padded;
      if (smp && m.direct) stage_unaligned<EB>(m, stage);
      else if (padded) pad_item_tail<EB>(stage, m.n);
      const int pslot = m.pslot, c = m.c;
      float2 pr;
      if (smp) {
        const float c_hi = m.c_hi, c_lo = m.c_lo;
        uint32_t w[kItemWords];
        const float mx = item_load_max<EB>(stage, w);
        if (written) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        ++processed;
        (void)top_up();  // the buffer's next copy runs during the exponentials
        pr = make_float2(mx, item_exp_sum<EB>(w, mx, c_hi, c_lo));
      } else {
        pr = a_item_greedy<EB>(m, stage);
        if (written) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        ++processed;
      }
      if (lane == 0) s_part(sl)[pslot * NC + c] = pr;
    } else {
      const unsigned long long sr = r_item<EB>(m, stage);
      if (lane == 0) s_rsum(sl)[m.c] = sr;
      __syncwarp();
      ++processed;
    }
    // the item is counted; the phase's last item runs what follows it
    __threadfence_block();
    unsigned int old = 0;
    if (lane == 0) old = atomicAdd(&ring[seq % kPipeRing].done, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    const bool last = old + 1 == ring[seq % kPipeRing].n;
    PipePhase ph;
    if (last) {
      __threadfence_block();
      ph = ring[seq % kPipeRing];
    }
    hold = INT_MAX;
    if (shown != pseq) {  // the cursor moved on while the item was processed
      __syncwarp();       // every lane has its copy of the record
      shown = pseq;
      if (lane == 0) *reinterpret_cast<volatile int*>(&s_pseq[warp]) = shown;
    }
    // this warp's copy in flight (if any) waits; the follow-up uses the
    // slot's own staging buffer
    if (last) follow(ph);
  }
  // copies still in flight are waited for (bounded)
  for (; processed != issued; ++processed) (void)mbar_wait(&bar[warp], processed & 1u, P.wait_ns);
  const unsigned int any = __reduce_or_sync(0xffffffffu, flags);
  if (lane == 0 && any) atomicOr(P.status, any);
  // the last CTA out resets the claim counter for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(P.exit_count, 1u) == gridDim.x - 1 ? 1 : 0;
  }
  __syncthreads();
  if (s_last && tid == 0) {
    *P.next_item = 0;
    *P.exit_count = 0;
    __threadfence();
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

// staging buffers, then rowpre [B+1] (padded to even), tconst [B] and cbase [B]
__host__ __device__ constexpr size_t smem_bytes(int B) {
  return (size_t)kWarps * kNB * kItemBytes + (size_t)((B + 2) & ~1) * sizeof(int) +
         (size_t)B * sizeof(TempC) + (size_t)B * sizeof(int);
}
constexpr size_t kMaxSmem = smem_bytes(kMaxBatch);
static_assert(kMaxSmem <= 227 * 1024 - 8 * 1024, "shared memory budget");

// Persistent grid: as many CTAs as fit on the device (cached per device).
template <int EB, int MODE, bool PK>
int grid_size() {
  static int cached_dev = -1, cached_grid = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev == cached_dev && cached_grid > 0) return cached_grid;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(verify_kernel<EB, MODE, PK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kMaxSmem) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<EB, MODE, PK>, kThreads,
                                                    kMaxSmem) != cudaSuccess)
    return 0;
  cached_dev = dev;
  cached_grid = sms * (per_sm > 0 ? per_sm : 1);
  return cached_grid;
}

// Schedule policy of the next calls (SV_SCHEDULE_*): AUTO takes the first of
// the resident cluster path, the streaming cluster path and the persistent
// grid that applies; STREAM skips the resident path; PERSISTENT forces the
// persistent grid (testing and benchmarking).
std::atomic<int> g_schedule{SV_SCHEDULE_AUTO};
// Limit of every bounded wait in the calls that follow (spec_verify_set_wait_limit).
std::atomic<unsigned long long> g_wait_ns{kWaitNs};
// Lazy positions on the request-claims path (spec_verify_set_lazy).
std::atomic<int> g_lazy{kLazyDefault};

size_t cluster_tables(int G, int V, int eb) {
  const size_t nc = ((size_t)V + kItemBytes / eb - 1) / (kItemBytes / eb);
  const size_t ncr = ((size_t)V + kHalfBytes / eb - 1) / (kHalfBytes / eb);
  return (size_t)(2 * G + 1) * nc * sizeof(float2) + ncr * kBlk * sizeof(unsigned long long) +
         sizeof(ClusterDec);
}

// Streaming cluster path: the partials and the leader's chunk sums.
size_t stream_tables(int G, int V, int eb) {
  const size_t nc = ((size_t)V + kItemBytes / eb - 1) / (kItemBytes / eb);
  const size_t ncr = ((size_t)V + kHalfBytes / eb - 1) / (kHalfBytes / eb);
  // partials [2G+1][NC], chunk sums [NCR], the bonus row's partials [NC]
  return (size_t)(2 * G + 2) * nc * sizeof(float2) + ncr * sizeof(unsigned long long);
}

// Clusters of C CTAs (C <= kClusterMax) of kernel `kern` that fit on this
// device at once, cached per device in cached[C] as (device + 1) << 16 | count
// (0: not yet known).  Also sets the kernel's shared-memory and cluster-size
// attributes for its launches.
template <class Kern>
int clusters_that_fit(Kern kern, int C, std::atomic<int>* cached, int threads = kThreads,
                      size_t smem = kClusterSmem) {
  int dev = 0;
  if (C < 1 || C > kClusterMax || cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int c0 = cached[C].load(std::memory_order_relaxed);
  if ((c0 >> 16) == dev + 1) return c0 & 0xffff;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
          cudaSuccess &&
      (C <= 8 || cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                     cudaSuccess)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned int)C);
    cfg.blockDim = dim3((unsigned int)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned int)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();  // a refused size only means that size is not used
  n = n < 0 ? 0 : (n > 0xffff ? 0xffff : n);
  cached[C].store(((dev + 1) << 16) | n, std::memory_order_relaxed);
  return n;
}

template <int EB, int MODE, bool PK>
int max_clusters(int C) {
  static std::atomic<int> cached[kClusterMax + 1];
  return clusters_that_fit(cluster_kernel<EB, MODE, PK>, C, cached);
}
// Shapes of the streaming kernel: warps and buffers per CTA, CTAs per SM.
// One wave of clusters (a request each) runs one CTA per SM; greedy claims
// run two CTAs per SM with half the warps each.  Sampling uses 16 warps per
// SM with one buffer each (the item is held in registers during its
// exponentials, 128 registers per thread); greedy, with light arithmetic,
// 12 warps with two buffers each.  A CTA's tables are capped so that its CTAs
// fit the SM's 228 KB of shared memory (1 KB of it reserved per CTA, about
// 3 KB of static shared memory each).
template <int MODE, int CPS>
struct StreamShape {
  static constexpr int nb = MODE == MODE_SAMPLE ? 1 : 2;
  static constexpr int nw = (MODE == MODE_SAMPLE ? 16 : kWarps) / CPS;
  static constexpr size_t table_cap =
      CPS == 1 ? (size_t)kClusterTables : (size_t)(CPS == 2 ? 12 : 8) * 1024;
  static constexpr size_t smem = (size_t)nw * nb * kItemBytes + table_cap;
  static_assert(CPS * (smem + 4 * 1024) <= 228 * 1024, "streaming CTAs per SM");
};
// Claimed requests: the claim order and the row counts it is built from.
// Sampling claims run one 16-warp CTA per SM: with the longest-first order
// they beat two 8-warp CTAs per SM (B=256 ragged: 127 against 177 us), whose
// CTA pairs share an SM's rate whatever their requests.  Greedy claims run two
// 6-warp CTAs per SM (B=512: 45 and 80 us against 48 and 83 with one CTA).
size_t claim_bytes(int B) { return ((size_t)B * 5 + 15) & ~(size_t)15; }
#ifndef SV_SAMPLE_CPS
#define SV_SAMPLE_CPS 1
#endif
#ifndef SV_GREEDY_CPS
#define SV_GREEDY_CPS 2  // three 4-warp CTAs per SM: B = 512 greedy 51.6 -> 58.8 us
#endif
template <int MODE>
constexpr int claim_cps() { return MODE == MODE_SAMPLE ? SV_SAMPLE_CPS : SV_GREEDY_CPS; }

template <int EB, int MODE, bool PK, int CPS>
int max_stream_clusters(int C) {
  using S = StreamShape<MODE, CPS>;
  static std::atomic<int> cached[kClusterMax + 1];
  return clusters_that_fit(stream_kernel<EB, MODE, PK, S::nw, S::nb, CPS>, C, cached, S::nw * 32,
                           S::smem);
}

// Resident cluster path: the cluster size for this call, or 0.
template <int EB, int MODE, bool PK>
int cluster_route(int B, int G, int V) {
  if (B < 1 || cluster_tables(G, V, EB) > (size_t)kClusterTables) return 0;
  const size_t nc = ((size_t)V + kItemBytes / EB - 1) / (kItemBytes / EB);
  // the largest cluster of which B fit at once (one wave: a request per
  // cluster) and whose warps hold one unit each of a request's A work
  for (int C = kClusterMax; C >= 8; --C)
    if (max_clusters<EB, MODE, PK>(C) >= B) return (size_t)(G + 1) * nc <= (size_t)C * kWarps ? C : 0;
  return 0;
}

template <int EB, int MODE, bool PK>
int launch_cluster(const Params& P, int C, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned int)(P.B * C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)kWarps * kNB * kItemBytes + cluster_tables(P.G, P.V, EB);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned int)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, cluster_kernel<EB, MODE, PK>, P) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

struct Route {
  int kind;  // SV_ROUTE_*
  int C;     // cluster size (cluster paths)
  int Q;     // clusters launched (cluster paths)
};

// Streaming cluster path: the largest cluster of which B fit at once (one
// wave, a request per cluster); with `claims`, a batch beyond one wave of
// single-CTA clusters runs on as many CTAs as fit, each claiming requests in
// turn.
template <int EB, int MODE, bool PK>
Route stream_route(int B, int G, int V) {
  const Route none{SV_ROUTE_PERSISTENT, 0, 0};
  if (B >= 1 && stream_tables(G, V, EB) <= StreamShape<MODE, 1>::table_cap)
    for (int C = kClusterMax; C >= 1; --C)
      if (max_stream_clusters<EB, MODE, PK, 1>(C) >= B) return Route{SV_ROUTE_STREAM, C, B};
  // beyond one wave: the streaming kernel's claims
  if (B < 1 || stream_tables(G, V, EB) > StreamShape<MODE, 1>::table_cap) return none;
  constexpr int QC = claim_cps<MODE>();
  if (stream_tables(G, V, EB) + claim_bytes(B) > StreamShape<MODE, QC>::table_cap) return none;
  const int Q = max_stream_clusters<EB, MODE, PK, QC>(1);
  return Q > 0 ? Route{SV_ROUTE_CLAIMS, 1, Q < B ? Q : B} : none;
}

#ifndef SV_PIPE
#define SV_PIPE 1
#endif
// The pipeline kernel's shared memory: buffers | per slot: partials, chunk
// sums, draw staging | claim order and row counts.
size_t pipe_smem(int B, int G, int V, int eb) {
  const size_t nc = ((size_t)V + kItemBytes / eb - 1) / (kItemBytes / eb);
  const size_t ncr = ((size_t)V + kHalfBytes / eb - 1) / (kHalfBytes / eb);
  const size_t part = ((size_t)(2 * G + 1) * nc * sizeof(float2) + 15) & ~(size_t)15;
  const size_t rsum = (ncr * sizeof(unsigned long long) + 15) & ~(size_t)15;
  return (size_t)kPipeWarps * kItemBytes + kPipeSlots * (part + rsum + kItemBytes) +
         (((size_t)B * 5 + 15) & ~(size_t)15);
}
constexpr size_t kPipeSmemCap = (size_t)200 * 1024;
// CTAs of the pipeline kernel that fit at once: one per SM (cached).
template <int EB, bool PK>
int pipe_ctas() {
  static std::atomic<int> cached{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int c0 = cached.load(std::memory_order_relaxed);
  if ((c0 >> 16) == dev + 1) return c0 & 0xffff;
  auto kern = pipe_kernel<EB, PK, kPipeWarps>;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPipeSmemCap) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPipeWarps * 32, kPipeSmemCap) !=
          cudaSuccess)
    per_sm = 0;
  (void)cudaGetLastError();
  int n = sms * (per_sm > 0 ? 1 : 0);
  n = n > 0xffff ? 0xffff : n;
  cached.store(((dev + 1) << 16) | n, std::memory_order_relaxed);
  return n;
}

template <int EB, int MODE, bool PK>
Route route(int B, int G, int V) {
  const int sched = g_schedule.load();
  if (sched == SV_SCHEDULE_PERSISTENT) return Route{SV_ROUTE_PERSISTENT, 0, 0};
  if (sched == SV_SCHEDULE_AUTO) {
    const int C = cluster_route<EB, MODE, PK>(B, G, V);
    if (C > 0) return Route{SV_ROUTE_CLUSTER, C, B};
  }
  // Beyond one wave, claimed requests (longest first) beat the persistent
  // grid's chunk claims: B=256 ragged, B=512 gamma 1 and 3, sampling 159 ->
  // 127, 142 -> 124, 225 -> 214 us; greedy 64 -> 64, 58 -> 45, 92 -> 80 us.
  // The grid remains for batches whose claim order does not fit.
  const Route r = stream_route<EB, MODE, PK>(B, G, V);
  if constexpr (MODE == MODE_SAMPLE) {
    // sampled claims with lazy positions (two requests or more per CTA): the
    // pipeline kernel (B = 512, gamma 3: 170.6 -> 153.8 us; gamma 1: 109.7 ->
    // 101.9 us)
    if (SV_PIPE && sched == SV_SCHEDULE_AUTO && r.kind == SV_ROUTE_CLAIMS && g_lazy.load() &&
        pipe_smem(B, G, V, EB) <= kPipeSmemCap) {
      const int Q = pipe_ctas<EB, PK>();
      if (Q > 0 && B >= 2 * Q) return Route{SV_ROUTE_PIPELINE, 1, Q};
    }
  }
  return r;
}

template <int EB, int MODE, bool PK, int CPS>
int launch_stream(const Params& P, int C, int Q, cudaStream_t stream) {
  using S = StreamShape<MODE, CPS>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned int)(Q * C));
  cfg.blockDim = dim3((unsigned int)(S::nw * 32));
  cfg.dynamicSmemBytes = (size_t)S::nw * S::nb * kItemBytes + stream_tables(P.G, P.V, EB) +
                         (Q * C < P.B ? claim_bytes(P.B) : 0);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned int)C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, stream_kernel<EB, MODE, PK, S::nw, S::nb, CPS>, P) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

template <int EB, int MODE, bool PK>
int launch(const Params& P, cudaStream_t stream) {
  const Route r = route<EB, MODE, PK>(P.B, P.G, P.V);
  if constexpr (MODE == MODE_SAMPLE) {
    if (r.kind == SV_ROUTE_PIPELINE) {
      pipe_kernel<EB, PK, kPipeWarps><<<r.Q, kPipeWarps * 32, pipe_smem(P.B, P.G, P.V, EB), stream>>>(P);
      return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
  }
  if (r.kind == SV_ROUTE_CLUSTER) return launch_cluster<EB, MODE, PK>(P, r.C, stream);
  if (r.kind == SV_ROUTE_STREAM) return launch_stream<EB, MODE, PK, 1>(P, r.C, r.Q, stream);
  if (r.kind == SV_ROUTE_CLAIMS) return launch_stream<EB, MODE, PK, claim_cps<MODE>()>(P, r.C, r.Q, stream);
  const int grid = grid_size<EB, MODE, PK>();
  if (grid <= 0) return SV_ERR_CUDA;
  // requests are processed in launches of at most kMaxBatch
  const int B = P.B;
  for (int b0 = 0; b0 < B; b0 += kMaxBatch) {
    Params Q = P;
    Q.B = B - b0 < kMaxBatch ? B - b0 : kMaxBatch;
    const size_t G = (size_t)P.G, V = (size_t)P.V;
    if (PK) {
      // packed: rows, tokens, uniforms and p/q are addressed through cu,
      // which keeps global offsets; only per-request arrays move
      Q.cu = P.cu + b0;
      Q.b_base = P.b_base + b0;
    } else {
      Q.target = P.target + (size_t)b0 * (G + 1) * V * EB;
      Q.draft = P.draft ? P.draft + (size_t)b0 * G * V * EB : nullptr;
      Q.tokens = P.tokens ? P.tokens + (size_t)b0 * G : nullptr;
      Q.uniforms = P.uniforms ? P.uniforms + (size_t)b0 * (G + 1) : nullptr;
      Q.p_tok = P.p_tok ? P.p_tok + (size_t)b0 * G : nullptr;
      Q.q_tok = P.q_tok ? P.q_tok + (size_t)b0 * G : nullptr;
    }
    Q.gamma = P.gamma ? P.gamma + b0 : nullptr;
    Q.temperature = P.temperature ? P.temperature + b0 : nullptr;
    Q.out_tokens = P.out_tokens + (size_t)b0 * (G + 1);
    Q.num_accepted = P.num_accepted ? P.num_accepted + b0 : nullptr;
    Q.cnt_a = P.cnt_a + b0;
    Q.cnt_r = P.cnt_r + b0;
    Q.dec = P.dec + b0;
    Q.queue = P.queue + b0;
    Q.stats = P.stats + (size_t)b0 * (2 * G + 1) * P.stride_nc;
    Q.resid = P.resid + (size_t)b0 * P.stride_ncr;
    const size_t smem = smem_bytes(Q.B);
    verify_kernel<EB, MODE, PK><<<grid, kThreads, smem, stream>>>(Q);
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
  P.cu = nullptr;
  P.total = 0;
  P.b_base = 0;
  P.uniforms = uniforms;
  P.temperature = temperature;
  P.out_tokens = out_tokens;
  P.num_accepted = num_accepted;
  P.p_tok = p_tok;
  P.q_tok = q_tok;
  P.status = reinterpret_cast<unsigned int*>(w + L.status);
  P.wait_ns = g_wait_ns.load();
  P.lazy = g_lazy.load();
  P.next_item = reinterpret_cast<unsigned int*>(w + L.next_item);
  P.exit_count = reinterpret_cast<unsigned int*>(w + L.exit_count);
  P.r_next = reinterpret_cast<unsigned int*>(w + L.r_next);
  P.q_tail = reinterpret_cast<unsigned int*>(w + L.q_tail);
  P.dec_count = reinterpret_cast<unsigned int*>(w + L.dec_count);
  P.cnt_a = reinterpret_cast<unsigned int*>(w + L.cnt_a);
  P.cnt_r = reinterpret_cast<unsigned int*>(w + L.cnt_r);
  P.dec = reinterpret_cast<DecRecord*>(w + L.dec);
  P.queue = reinterpret_cast<DecRecord*>(w + L.queue);
  P.stats = reinterpret_cast<float2*>(w + L.stats);
  P.resid = reinterpret_cast<unsigned long long*>(w + L.resid);
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
  return dtype == SV_BF16 ? launch<2, MODE_SAMPLE, false>(P, s)
                          : launch<4, MODE_SAMPLE, false>(P, s);
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
  return dtype == SV_BF16 ? launch<2, MODE_GREEDY, false>(P, s)
                          : launch<4, MODE_GREEDY, false>(P, s);
}

int spec_verify_sample_packed(const void* target_logits, const void* draft_logits,
                              sv_dtype dtype, int B, int G, int V, const int32_t* cu_draft,
                              int total_drafts, const int32_t* draft_tokens,
                              const float* uniforms, const float* temperature,
                              int32_t* out_tokens, int32_t* num_accepted, double* p_tok,
                              double* q_tok, void* workspace, size_t ws_bytes,
                              sv_stream_t stream) {
  int rc = check_scalars(dtype, B, G, V);
  if (rc) return rc;
  if (total_drafts < 0) return SV_ERR_SCALAR;
  if (!target_logits || !cu_draft || !uniforms || !temperature || !out_tokens ||
      !num_accepted || !workspace)
    return SV_ERR_NULL;
  if (total_drafts > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_NULL;
  if (!aligned(cu_draft, 4)) return SV_ERR_ALIGN;
  Params P;
  rc = fill_params(P, target_logits, draft_logits, dtype, B, G, V, draft_tokens, nullptr,
                   uniforms, temperature, out_tokens, num_accepted, p_tok, q_tok, workspace,
                   ws_bytes);
  if (rc) return rc;
  P.cu = cu_draft;
  P.total = total_drafts;
  if (B == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == SV_BF16 ? launch<2, MODE_SAMPLE, true>(P, s)
                          : launch<4, MODE_SAMPLE, true>(P, s);
}

int spec_verify_greedy_packed(const void* target_logits, sv_dtype dtype, int B, int G, int V,
                              const int32_t* cu_draft, int total_drafts,
                              const int32_t* draft_tokens, int32_t* out_tokens,
                              int32_t* num_accepted, void* workspace, size_t ws_bytes,
                              sv_stream_t stream) {
  int rc = check_scalars(dtype, B, G, V);
  if (rc) return rc;
  if (total_drafts < 0) return SV_ERR_SCALAR;
  if (!target_logits || !cu_draft || !out_tokens || !num_accepted || !workspace)
    return SV_ERR_NULL;
  if (total_drafts > 0 && !draft_tokens) return SV_ERR_NULL;
  if (!aligned(cu_draft, 4)) return SV_ERR_ALIGN;
  Params P;
  rc = fill_params(P, target_logits, nullptr, dtype, B, G, V, draft_tokens, nullptr, nullptr,
                   nullptr, out_tokens, num_accepted, nullptr, nullptr, workspace, ws_bytes);
  if (rc) return rc;
  P.cu = cu_draft;
  P.total = total_drafts;
  if (B == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == SV_BF16 ? launch<2, MODE_GREEDY, true>(P, s)
                          : launch<4, MODE_GREEDY, true>(P, s);
}

int spec_verify_draw(const void* logits, sv_dtype dtype, int B, int V, const float* uniforms,
                     const float* temperature, int32_t* tokens, void* workspace, size_t ws_bytes,
                     sv_stream_t stream) {
  int rc = check_scalars(dtype, B, 0, V);
  if (rc) return rc;
  if (!logits || !uniforms || !temperature || !tokens || !workspace) return SV_ERR_NULL;
  // the sampling step with no drafts: each row's bonus draw
  Params P;
  rc = fill_params(P, logits, nullptr, dtype, B, 0, V, nullptr, nullptr, uniforms, temperature,
                   tokens, nullptr, nullptr, nullptr, workspace, ws_bytes);
  if (rc) return rc;
  if (B == 0) return SV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return dtype == SV_BF16 ? launch<2, MODE_SAMPLE, false>(P, s)
                          : launch<4, MODE_SAMPLE, false>(P, s);
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
  // counters, arrival counts and decision records start at zero for every call
  if (cudaMemsetAsync(ws, 0, L.stats, s) != cudaSuccess) return SV_ERR_CUDA;
  return dtype == SV_BF16 ? launch<2, MODE_SAMPLE, false>(P, s)
                          : launch<4, MODE_SAMPLE, false>(P, s);
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

int spec_verify_set_schedule(int schedule) {
  if (schedule != SV_SCHEDULE_AUTO && schedule != SV_SCHEDULE_PERSISTENT &&
      schedule != SV_SCHEDULE_STREAM)
    return SV_ERR_SCALAR;
  return g_schedule.exchange(schedule);
}

unsigned long long spec_verify_set_wait_limit(unsigned long long ns) {
  if (ns == 0ull) ns = kWaitNs;
  return g_wait_ns.exchange(ns);
}

int spec_verify_set_lazy(int on) {
  if (on != 0 && on != 1) return SV_ERR_SCALAR;
  return g_lazy.exchange(on);
}

int spec_verify_route(sv_dtype dtype, int B, int G, int V, int greedy, int* cluster_size) {
  const int rc = check_scalars(dtype, B, G, V);
  if (rc) return rc;
  Route r{SV_ROUTE_PERSISTENT, 0, 0};
  if (B > 0) {
    if (dtype == SV_BF16)
      r = greedy ? route<2, MODE_GREEDY, false>(B, G, V) : route<2, MODE_SAMPLE, false>(B, G, V);
    else
      r = greedy ? route<4, MODE_GREEDY, false>(B, G, V) : route<4, MODE_SAMPLE, false>(B, G, V);
  }
  if (cluster_size) *cluster_size = r.C;
  return r.kind;
}

int spec_verify_cluster_size(sv_dtype dtype, int B, int G, int V, int greedy) {
  int C = 0;
  const int rc = spec_verify_route(dtype, B, G, V, greedy, &C);
  return rc < 0 ? rc : C;
}

}  // extern "C"
