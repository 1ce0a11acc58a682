// Decode attention, split-K partials stage: persistent tensor-core kernel with
// shared-memory lookup-table dequantization.
//
// [P4] riverfrot.github.io "TurboQuant란 무엇이며…", §2.2 (decode: one query per
// head against every cached key, softmax, weighted sum of values), §4.2 (the
// codebook is only looked up at run time), §4.3 (stage-1 score plus the 1-bit
// QJL correction; softmax(QK^T/sqrt(d))); [P2] "생각정리 209 (TurboQuant)", stage 2.
//
// One CTA of 12 or 16 warps per SM (chosen per launch).  A work item is one
// (sequence, KV head, chunk); each warp takes items from a global counter and
// streams their 16-token pages through its own ring of 3-4 stages
// (cp.async.bulk, mbarrier completion); the ring runs on across item
// boundaries, so a warp never drains between items.
//
// Dequantization is a table lookup: one byte of packed codes (two codes) indexes
// a table whose entry is the fp16 pair of their centroids.  Each entry is
// replicated for the 32 lanes (entry e, lane l at byte 256 e + 4 l, K table at
// +0, V table at +128), so a warp's 32 lookups hit 32 different banks, and one
// prmt builds the address (the code byte as byte 1, the lane offset as byte 0).
// Keys pair two channels of one token (the byte as stored); values pair one
// channel of two consecutive tokens (two tokens' codes interleaved by lop3),
// the layout the value MMA wants.  3-bit octets are first gathered into eight
// nibbles (channels 6 and 7 sit in the spare bit of each nibble).
//   * scores: S1 = K^ Q~^T and S2 = (1 + c b) U^T, m16n8k16 with the 16 tokens on
//     M and the G <= 8 query heads of the KV head on N (K = channels, or the m
//     projections); the sign bits b become fp16 1 or 1 + c (c = 255/1024) by one
//     prmt per pair, and <u, 2b - 1> = (2/c) S2 - (2/c + 1) sum(u);
//   * logits = (n_k/sqrt(d) S1 + sqrt(pi/2)/m rho S2) * scale; online softmax
//     on the accumulator fragments;
//   * P' = p * n_v / sqrt(d), transposed in registers (movmatrix) into the B
//     operand of O^T += V^^T P'^T (M = channels, K = tokens).
// The channel order inside the fragments is a fixed permutation that makes each
// thread's code bytes contiguous; Q~ and the output use the same permutation.
//
// Supported here: d = 128, m = 128, channel split 64, the bit-width
// combinations instantiated below.  Other configurations run the CUDA-core
// kernel in tq_decode.cu.

#include "tq_internal.h"

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {
namespace {

// Warps per CTA: 16, or 12 with deeper rings and up to 168 registers per
// thread; lut_warps_for picks per launch (tq_internal.h).
constexpr int kMaxStagesL = 4;         // ring depth per warp: the largest <= this that fits
constexpr float kInvSqrtD = 0.08838834764831845f;
constexpr float kSqrtHalfPi = 1.2533141373155003f;
constexpr int kWaitLimit = 1 << 22;
constexpr float kNegBig = -1.0e30f;    // finite "minus infinity": 2^(kNegBig - m) is exactly 0, never NaN
// Slack of the running softmax max (log2 units): p <= 8, and 8 * 65504 / sqrt(128)
// is below the fp16 maximum, so no fp16 value norm can overflow P'.
constexpr float kLazyMax = 3.0f;
constexpr int kSmemLimit = 232448;     // opt-in shared memory per block

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Bounded wait for phase `parity`; false after kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 2^x (ex2.approx.ftz: about 2 ulp; the finite -1e30 sentinel gives exactly 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t f16bits(float x) { return __half_as_ushort(__float2half_rn(x)); }
// (lo, hi) as an fp16 pair, each rounded to nearest even.
__device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Transpose of an 8x8 fp16 matrix held as one pair per lane (lane 4r + c: row r,
// columns 2c, 2c + 1), returned in the same layout.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) { return f16bits(lo) | (f16bits(hi) << 16); }

// ---------------------------------------------------------------------------
// tables
// ---------------------------------------------------------------------------
// Entries used per bit width: 4-bit bytes 0..255; 3-bit gathered nibble pairs
// 0x00..0x77; 2-bit nibbles (two 2-bit codes) 0..15.
__host__ __device__ constexpr int lut_entries(int b) { return b == 4 ? 256 : b == 3 ? 120 : 16; }
__host__ __device__ constexpr int region_bytes(int kb, int vb) {
  return 256 * (lut_entries(kb) > lut_entries(vb) ? lut_entries(kb) : lut_entries(vb));
}

// Code of a stored field value (4-bit fields are sign-magnitude, see tq.h).
__device__ __forceinline__ int stored_code(int b, int f) { return b == 4 ? (f < 8 ? f + 8 : 15 - f) : f; }

// fp16 pair of the centroids of the two fields of index e.
__device__ uint32_t lut_entry(const GroupBook& gb, int b, int e) {
  const int w = b == 2 ? 2 : 4;
  const int mask = b == 4 ? 15 : b == 3 ? 7 : 3;
  return pack_h2(gb.c[stored_code(b, e & mask)], gb.c[stored_code(b, (e >> w) & mask)]);
}

// 3-bit octet (24 bits as stored) -> eight nibbles, nibble i = code of channel i.
// Channels 0-5 sit in nibbles already; the spare bits 3/11/19 (channel 6) and
// 7/15/23 (channel 7) are gathered to bits 24-26 and 28-30 by one multiply.
__device__ __forceinline__ uint32_t gather_octet(uint32_t v) {
  return (v & 0x00777777u) | (((v & 0x00888888u) * 0x00204080u) & 0x77000000u);
}

__device__ __forceinline__ uint32_t bits_at(const uint32_t* w, int off) {
  return __funnelshift_r(w[off >> 5], w[(off >> 5) + 1], off & 31);
}

// The eight key pair indices of thread slice t (channels 16t..16t+15 of a
// group): pair j is byte j&3 of x[j>>2].
template <int B>
__device__ __forceinline__ void k_slice(const uint32_t* grp, int t, uint32_t (&x)[2]) {
  if (B == 4) {
    const uint2 w = reinterpret_cast<const uint2*>(grp)[t];
    x[0] = w.x;
    x[1] = w.y;
  } else if (B == 3) {
    x[0] = gather_octet(bits_at(grp, 48 * t));
    x[1] = gather_octet(bits_at(grp, 48 * t + 24));
  } else {
    const uint32_t w = grp[t];
    x[0] = w & 0x0F0F0F0Fu;
    x[1] = (w >> 4) & 0x0F0F0F0Fu;
  }
}
// (k_pair_channel in tq_internal.h gives the channel of the low half of pair j.)

// Codes of channels 8g..8g+7 of one value vector (group-relative words).
template <int B>
__device__ __forceinline__ uint32_t v_word(const uint32_t* grp, int g) {
  if (B == 4) return grp[g];
  if (B == 3) return gather_octet(bits_at(grp, 24 * g));
  return (grp[g >> 1] >> (16 * (g & 1))) & 0xFFFFu;
}
// Token-pair indices of the eight channels from the words of tokens a and a+1:
// m-tile mt uses byte mt&3 of (mt < 4 ? lo : hi).
template <int B>
__device__ __forceinline__ void v_pairs(uint32_t xa, uint32_t xb, uint32_t& lo, uint32_t& hi) {
  if (B == 2) {
    const uint32_t A = (xa & 0x3333u) | ((xb << 2) & 0xCCCCu);
    const uint32_t Bm = ((xa >> 2) & 0x3333u) | (xb & 0xCCCCu);
    const uint32_t C = A | (Bm << 16);
    lo = C & 0x0F0F0F0Fu;
    hi = (C >> 4) & 0x0F0F0F0Fu;
  } else {
    lo = (xa & 0x0F0F0F0Fu) | ((xb << 4) & 0xF0F0F0F0u);
    hi = ((xa >> 4) & 0x0F0F0F0Fu) | (xb & 0xF0F0F0F0u);
  }
}
// Channel (within the eight) that m-tile mt covers.
__host__ __device__ constexpr int v_channel(int b, int mt) {
  return b == 2 ? (mt == 0 ? 0 : mt == 1 ? 4 : mt == 2 ? 1 : mt == 3 ? 5 : mt == 4 ? 2 : mt == 5 ? 6 : mt == 6 ? 3 : 7)
                : (mt < 4 ? 2 * mt : 2 * (mt - 4) + 1);
}

// QJL sign pair for the MMA from xs = w << (7 - s): bits s + 16h and s + 8 + 16h
// of the sign word w as the fp16 pair (1 + kQjlC b, 1 + kQjlC b'), b = bit:
// prmt's sign-replicate selectors copy a byte's top bit into the low byte of
// each half (0xFF or 0), the high byte is 0x3C (1.0).
constexpr float kQjlC = 255.0f / 1024.0f;
__device__ __forceinline__ uint32_t qjl_pair(uint32_t xs, int h) {
  return prmt(xs, 0x3C3C3C3Cu, h ? 0x4B4Au : 0x4948u);
}

struct Slot {
  int item;    // -1: no more work
  int page;    // page index within the item's chunk
  int valid;   // 0: page id out of range (flagged), no data
  int pad;
};

template <int W, int KBH, int KBL, int VBH, int VBL, bool QJL>
struct Geo {
  static constexpr int CBK = (64 * KBH + 64 * KBL) / 8;
  static constexpr int CBV = (64 * VBH + 64 * VBL) / 8;
  static constexpr int KBB = 16 * (CBK + (QJL ? 16 + 2 : 0) + 2);
  static constexpr int VBB = 16 * (CBV + 2);
  static constexpr int STAGE = KBB + VBB;
  static constexpr int K_SIGNS = 16 * CBK;
  static constexpr int K_NORM = K_SIGNS + (QJL ? 16 * 16 : 0);
  static constexpr int K_RNORM = K_NORM + 32;
  static constexpr int V_NORM = 16 * CBV;
  static constexpr int R0 = region_bytes(KBH, VBH);
  static constexpr int R1 = region_bytes(KBL, VBL);
  static constexpr int TABLES = R0 + R1;
  // per warp: ring, then (in the extras block) S barriers and S slots
  __host__ __device__ static constexpr int extras(int st) { return W * (st * 8 + st * 16); }
  // the tables start at a 64 KiB-aligned shared address; the gap below them
  // takes whole warp rings, so at most one ring (or, when every ring fits in
  // the gap, the rest of the gap) is lost to the alignment
  __host__ __device__ static constexpr int rings_plus_gap(int st) {
    return (W + 1) * st * STAGE > 65536 ? (W + 1) * st * STAGE : 65536;
  }
  __host__ __device__ static constexpr int need(int st) { return TABLES + rings_plus_gap(st) + extras(st) + 1024; }
  static constexpr int STAGES = need(kMaxStagesL) <= kSmemLimit ? kMaxStagesL
                                : need(kMaxStagesL - 1) <= kSmemLimit ? kMaxStagesL - 1
                                : need(3) <= kSmemLimit ? 3 : 2;
  static constexpr int RINGW = STAGES * STAGE;
  static constexpr int SMEM = need(STAGES);
  static_assert(STAGE % 16 == 0 && TABLES % 256 == 0, "bulk copy alignment");
  static_assert(SMEM <= kSmemLimit, "shared memory per block");
};

// Shared load at a full 32-bit shared address plus a constant offset.
template <int OFF>
__device__ __forceinline__ uint32_t lds_at(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int W, int KBH, int KBL, int VBH, int VBL, bool QJL, bool CAUSAL = false>
__global__ void __launch_bounds__(32 * W, 1) lut_partials_kernel(DecodeArgs a, int total_items) {
  using Gm = Geo<W, KBH, KBL, VBH, VBL, QJL>;
  constexpr int S = Gm::STAGES;
  // the merge after this kernel may launch now: it stages what it can and then
  // waits for this grid; persistent CTAs are all resident, so none is delayed
  pdl_trigger();
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  // ---- layout: tables at the first 64 KiB boundary, rings around them ------
  const uint32_t base = smem_u32(smem);
  const uint32_t tab = (base + 0xFFFFu) & ~0xFFFFu;
  const int n_low = min(W, static_cast<int>((tab - base) / Gm::RINGW));   // rings below the tables
  const uint32_t ext = tab + Gm::TABLES + (W - n_low) * Gm::RINGW;
  if (ext + Gm::extras(S) > base + Gm::SMEM) {          // cannot happen with the sizes above
    if (threadIdx.x == 0) atomicOr(a.tab.err, kErrLayout);
    return;
  }
  auto at = [&](uint32_t addr) { return smem + (addr - base); };
  // ---- tables (once per CTA) ------------------------------------------------
  {
    constexpr int E0 = Gm::R0 / 256, E1 = Gm::R1 / 256;
    for (int i = threadIdx.x; i < (E0 + E1) * 16; i += 32 * W) {
      const int quad = i & 7, which = (i >> 3) & 1;
      int e = i >> 4;
      const int region = e < E0 ? 0 : 1;
      if (region) e -= E0;
      const int b = region ? (which ? VBL : KBL) : (which ? VBH : KBH);
      const GroupBook& gb = (which ? a.vl : a.kl).g[region];
      const uint32_t v = e < lut_entries(b) ? lut_entry(gb, b, e) : 0u;
      *reinterpret_cast<uint4*>(at(tab + (region ? Gm::R0 : 0) + e * 256 + which * 128 + quad * 16)) =
          make_uint4(v, v, v, v);
    }
  }
  unsigned char* ring = at(warp < n_low ? base + warp * Gm::RINGW : tab + Gm::TABLES + (warp - n_low) * Gm::RINGW);
  unsigned long long* bars = reinterpret_cast<unsigned long long*>(at(ext)) + warp * S;
  Slot* slots = reinterpret_cast<Slot*>(at(ext + W * S * 8)) + warp * S;
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_u32(&bars[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int nch = a.nchunks, C = a.chunk;
  auto seq_len = [&](int b) {
    int L = a.seq_lens[b] + a.len_add;
    if (L < 0 || L > a.max_seq_len || L > a.maxp * kPage) {
      atomicOr(a.tab.err, kErrSeqLen);
      L = L < 0 ? 0 : L;
      L = L > a.max_seq_len ? a.max_seq_len : L;
      L = L > a.maxp * kPage ? a.maxp * kPage : L;
    }
    return L;
  };

  // causal: query rows of a (sequence, KV head) are r = t G + g (new token t,
  // query head g of the group), eight per block; row r attends positions
  // [0, seq_lens[b] + t] (seq_lens holds the first new position, len_add = T).
  // block_len: the positions any row of block qb needs; row_len: one row's.
  auto row_len = [&](int b, int r) {
    if (r >= a.T * a.G) return 0;
    const int L = a.seq_lens[b] + r / a.G + 1;
    return min(L, seq_len(b));
  };
  auto block_len = [&](int b, int qb) {
    const int last = min(a.T * a.G - 1, 8 * qb + 7);
    return row_len(b, last);
  };

  // ---- producer state (meaningful in lane 0) --------------------------------
  int p_item = 0, p_page = 0, p_npages = 0, p_b = 0, p_h = 0, p_chunk = 0;   // p_item -1: done
  int p_pid = 0;                 // page id of (p_item, p_page), loaded one refill ahead
  const int* p_row = a.block_table;
  auto issue = [&](int s) {      // lane 0: fill slot s with the next page of this warp's stream
    const uint32_t bar = smem_u32(&bars[s]);
    while (p_item >= 0 && p_page >= p_npages) {
      const int it = atomicAdd(a.sched, 1);
      if (it >= total_items) {
        p_item = -1;
        break;
      }
      p_chunk = it % nch;
      const int rest = it / nch;
      const int bh = CAUSAL ? rest / a.nqb : rest;
      p_h = bh % a.H;
      p_b = bh / a.H;
      const int L = CAUSAL ? block_len(p_b, rest % a.nqb) : seq_len(p_b);
      const int t0 = p_chunk * C;
      if (t0 >= L) continue;                  // chunk past the end: no partial (the merge skips it)
      p_item = it;
      p_page = 0;
      p_npages = (min(t0 + C, L) - t0 + kPage - 1) / kPage;
      p_row = a.block_table + static_cast<long long>(p_b) * a.maxp + p_chunk * (C / kPage);
      p_pid = p_row[0];
    }
    Slot& sl = slots[s];
    if (p_item < 0) {
      sl.item = -1;
      sl.valid = 0;
      mbar_arrive(bar);
      return;
    }
    sl.item = p_item;
    sl.page = p_page;
    const int page = p_pid;
    ++p_page;
    if (page < 0 || page >= a.num_pages) {
      atomicOr(a.tab.err, kErrPage);
      sl.valid = 0;
      mbar_arrive(bar);
    } else {
      sl.valid = 1;
      unsigned char* dst = ring + s * Gm::STAGE;
      fence_proxy_async();
      mbar_arrive_tx(bar, Gm::STAGE);
      bulk_g2s(smem_u32(dst),
               a.kc + static_cast<long long>(page) * a.k_page_bytes + static_cast<long long>(p_h) * Gm::KBB, Gm::KBB,
               bar);
      bulk_g2s(smem_u32(dst + Gm::KBB),
               a.vc + static_cast<long long>(page) * a.v_page_bytes + static_cast<long long>(p_h) * Gm::VBB, Gm::VBB,
               bar);
    }
    // the next page id, loaded after the fence and arrive above (which wait for
    // this thread's outstanding memory operations) and used one refill later
    if (p_page < p_npages) p_pid = p_row[p_page];
  };
  // the query prep (the kernel before this one) zeroes the work counter and
  // writes the query fragments: everything above ran while it finished
  pdl_wait();
  if (lane == 0)
    for (int s = 0; s < S; ++s) issue(s);
  __syncwarp();

  // ---- consumer state ---------------------------------------------------------
  // prmt operand: byte 0 = lane offset (+128 for the V half), bytes 2-3 = the
  // 64 KiB block of the table region; byte 1 comes from the code byte
  constexpr int OFF1 = Gm::R0 & 0xFFFF;                      // region 1 offset inside its 64 KiB block
  const uint32_t lbk0 = tab | (static_cast<uint32_t>(lane) * 4u), lbv0 = lbk0 + 128u;
  const uint32_t lbk1 = lbk0 + (static_cast<uint32_t>(Gm::R0) & ~0xFFFFu), lbv1 = lbk1 + 128u;
  const float k1 = kInvSqrtD * a.scale_log2;
  const float k2 = kSqrtHalfPi / 128.0f * a.scale_log2;
  int cur = -1, c_b = 0, c_h = 0, c_chunk = 0, c_t0 = 0, c_t1 = 0, c_qb = 0;
  int c_end[2] = {0, 0};   // causal: end of the valid positions of this thread's columns 2t, 2t + 1
  const uint4* c_qlo = nullptr;   // fp16 low parts of this lane's q~ fragments (read per page, from L1)
  uint32_t qf[16], uf[16];
  float kqa, kqb[2];       // QJL logit terms: <u, +-1> = (2/c) raw - (2/c + 1) sum(u), times k2
  float acc[8][4];
  float m_run[2], l_run[2];
  bool failed = false;

  auto flush = [&]() {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float l = l_run[c];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int hh = 2 * t + c;
      const int r = 8 * c_qb + hh;
      if (CAUSAL ? r < a.T * a.G : hh < a.G) {
        const long long qrow = CAUSAL ? (static_cast<long long>(c_b) * a.T + r / a.G) * a.Hq + c_h * a.G + r % a.G
                                      : static_cast<long long>(c_b) * a.Hq + c_h * a.G + hh;
        float* dst = a.part + (qrow * nch + c_chunk) * (kD + 2);
        if (g == 0) {
          dst[0] = m_run[c];
          dst[1] = l;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          dst[2 + 8 * g + v_channel(VBH, mt)] = acc[mt][c];
          dst[2 + 64 + 8 * g + v_channel(VBL, mt)] = acc[mt][c + 2];
        }
      }
    }
  };
  auto start = [&](int item) {
    c_chunk = item % nch;
    const int rest = item / nch;
    const int bh = CAUSAL ? rest / a.nqb : rest;
    c_qb = CAUSAL ? rest % a.nqb : 0;
    c_h = bh % a.H;
    c_b = bh / a.H;
    c_t0 = c_chunk * C;
    c_t1 = min(c_t0 + C, CAUSAL ? block_len(c_b, c_qb) : seq_len(c_b));
    if (CAUSAL) {
      c_end[0] = min(c_t1, row_len(c_b, 8 * c_qb + 2 * t));
      c_end[1] = min(c_t1, row_len(c_b, 8 * c_qb + 2 * t + 1));
    }
    // the query fragments, packed by qprep in this thread's order: 8 x 16 B
    const int qr = 8 * c_qb + g;
    if (CAUSAL ? qr < a.T * a.G : g < a.G) {
      const long long qrow = CAUSAL ? (static_cast<long long>(c_b) * a.T + qr / a.G) * a.Hq + c_h * a.G + qr % a.G
                                    : static_cast<long long>(c_b) * a.Hq + c_h * a.G + g;
      const uint4* fp = reinterpret_cast<const uint4*>(a.qfrag + qrow * kQFragWords + 32 * t);
      c_qlo = reinterpret_cast<const uint4*>(a.qfrag + qrow * kQFragWords + 128 + 16 * t);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 x = fp[v], y = fp[4 + v];
        qf[4 * v] = x.x, qf[4 * v + 1] = x.y, qf[4 * v + 2] = x.z, qf[4 * v + 3] = x.w;
        uf[4 * v] = QJL ? y.x : 0u, uf[4 * v + 1] = QJL ? y.y : 0u;
        uf[4 * v + 2] = QJL ? y.z : 0u, uf[4 * v + 3] = QJL ? y.w : 0u;
      }
    } else {
#pragma unroll
      for (int v = 0; v < 16; ++v) qf[v] = uf[v] = 0u;
      c_qlo = nullptr;
    }
    if (QJL) {
      // sum of head g's u (the fp16 values the MMA multiplies), then the sums
      // of heads 2t, 2t+1 for this thread's accumulator columns
      float su = 0.0f;
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&uf[v]));
        su += f.x + f.y;
      }
      su += __shfl_xor_sync(0xffffffffu, su, 1);
      su += __shfl_xor_sync(0xffffffffu, su, 2);
      const float su0 = __shfl_sync(0xffffffffu, su, (2 * t) << 2);
      const float su1 = __shfl_sync(0xffffffffu, su, (2 * t + 1) << 2);
      kqa = k2 * (2.0f / kQjlC);
      kqb[0] = -k2 * (2.0f / kQjlC + 1.0f) * su0;
      kqb[1] = -k2 * (2.0f / kQjlC + 1.0f) * su1;
    } else {
      kqa = kqb[0] = kqb[1] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
    m_run[0] = m_run[1] = kNegBig;
    l_run[0] = l_run[1] = 0.0f;
  };

  // a warp consumes at most one slot per page of the launch plus its end
  // marker; more means a broken stream: flag it and stop
  const long long max_slots = static_cast<long long>(total_items) * (C / kPage) + S;
  int i = 0, drain_from = 1;
  for (;; ++i) {
    const int s = i % S;
    if (i > max_slots) {
      failed = true;
      drain_from = 0;
      if (lane == 0) atomicOr(a.tab.err, kErrTimeout);
      break;
    }
    // every lane polls; the vote makes a give-up uniform across the warp
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[s]), (i / S) & 1))) {
      failed = true;
      if (lane == 0) atomicOr(a.tab.err, kErrTimeout);
      break;
    }
    const Slot sl = slots[s];
    if (sl.item < 0) {                     // end of this warp's stream
      if (cur >= 0) flush();
      break;
    }
    if (sl.item != cur) {
      if (cur >= 0) flush();
      cur = sl.item;
      start(cur);
    }
    if (sl.valid) {
      const unsigned char* kb = ring + s * Gm::STAGE;
      const unsigned char* vb = kb + Gm::KBB;
      const int pbase = c_t0 + sl.page * kPage;
      // ---- scores ---------------------------------------------------------
      // two accumulators per score (channel group / even-odd projection
      // steps) halve the dependent HMMA chains
      float s1[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
      float s1b[4] = {0.f, 0.f, 0.f, 0.f}, s2b[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint32_t* ra = reinterpret_cast<const uint32_t*>(kb + g * Gm::CBK);
        const uint32_t* rb = reinterpret_cast<const uint32_t*>(kb + (g + 8) * Gm::CBK);
        uint32_t xa0[2], xb0[2], xa1[2], xb1[2];
        k_slice<KBH>(ra, t, xa0);
        k_slice<KBH>(rb, t, xb0);
        k_slice<KBL>(ra + 2 * KBH, t, xa1);
        k_slice<KBL>(rb + 2 * KBH, t, xb1);
        // causal attention (many queries per page, a heavier contraction): q~ =
        // hi + lo, the low parts (about 2^-11 of q~) through the same key
        // fragments into the other accumulator chain, halving the logit's
        // rounding error; decode keeps q~ in fp16 alone
        uint4 ql = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int kk = (q >> 1) + 4 * (q & 1);   // alternate the two channel groups
          const int j0 = 2 * (kk & 3), j1 = j0 + 1;
          const uint32_t* xa = kk < 4 ? xa0 : xa1;
          const uint32_t* xb = kk < 4 ? xb0 : xb1;
          const uint32_t s0 = 0x7604u | (static_cast<uint32_t>(j0 & 3) << 4);
          const uint32_t s1x = 0x7604u | (static_cast<uint32_t>(j1 & 3) << 4);
          uint32_t a0, a1, a2, a3;
          if (kk < 4) {
            a0 = lds_at<0>(prmt(xa[j0 >> 2], lbk0, s0));
            a1 = lds_at<0>(prmt(xb[j0 >> 2], lbk0, s0));
            a2 = lds_at<0>(prmt(xa[j1 >> 2], lbk0, s1x));
            a3 = lds_at<0>(prmt(xb[j1 >> 2], lbk0, s1x));
          } else {
            a0 = lds_at<OFF1>(prmt(xa[j0 >> 2], lbk1, s0));
            a1 = lds_at<OFF1>(prmt(xb[j0 >> 2], lbk1, s0));
            a2 = lds_at<OFF1>(prmt(xa[j1 >> 2], lbk1, s1x));
            a3 = lds_at<OFF1>(prmt(xb[j1 >> 2], lbk1, s1x));
          }
          mma16816(kk < 4 ? s1 : s1b, a0, a1, a2, a3, qf[2 * kk], qf[2 * kk + 1]);
          if (CAUSAL) {
            if ((kk & 1) == 0) ql = c_qlo ? __ldg(c_qlo + (kk >> 1)) : make_uint4(0u, 0u, 0u, 0u);
            mma16816(kk < 4 ? s1b : s1, a0, a1, a2, a3, (kk & 1) ? ql.z : ql.x, (kk & 1) ? ql.w : ql.y);
          }
        }
        if (QJL) {
          const uint32_t* sg = reinterpret_cast<const uint32_t*>(kb + Gm::K_SIGNS);
          const uint32_t wa = sg[g * 4 + t], wb = sg[(g + 8) * 4 + t];
#pragma unroll
          for (int st = 0; st < 8; ++st) {
            const uint32_t xa = wa << (7 - st), xb = wb << (7 - st);
            mma16816((st & 1) ? s2b : s2, qjl_pair(xa, 0), qjl_pair(xb, 0), qjl_pair(xa, 1), qjl_pair(xb, 1),
                     uf[2 * st], uf[2 * st + 1]);
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          s1[r] += s1b[r];
          s2[r] += s2b[r];
        }
      }
      const __half* nk = reinterpret_cast<const __half*>(kb + Gm::K_NORM);
      const __half* rk = reinterpret_cast<const __half*>(kb + Gm::K_RNORM);
      const __half* nv = reinterpret_cast<const __half*>(vb + Gm::V_NORM);
      const bool vg = pbase + g < c_t1;
      const bool vg8 = pbase + g + 8 < c_t1;
      float lg[4];
      {
        const float nkg = __half2float(nk[g]), nkg8 = __half2float(nk[g + 8]);
        const float rkg = QJL ? __half2float(rk[g]) : 0.f, rkg8 = QJL ? __half2float(rk[g + 8]) : 0.f;
        // causal: token p of column c is valid below that column's end
        const bool v0 = CAUSAL ? pbase + g < c_end[0] : vg, v1 = CAUSAL ? pbase + g < c_end[1] : vg;
        const bool v2 = CAUSAL ? pbase + g + 8 < c_end[0] : vg8, v3 = CAUSAL ? pbase + g + 8 < c_end[1] : vg8;
        lg[0] = v0 ? fmaf(nkg * k1, s1[0], rkg * fmaf(kqa, s2[0], kqb[0])) : kNegBig;
        lg[1] = v1 ? fmaf(nkg * k1, s1[1], rkg * fmaf(kqa, s2[1], kqb[1])) : kNegBig;
        lg[2] = v2 ? fmaf(nkg8 * k1, s1[2], rkg8 * fmaf(kqa, s2[2], kqb[0])) : kNegBig;
        lg[3] = v3 ? fmaf(nkg8 * k1, s1[3], rkg8 * fmaf(kqa, s2[3], kqb[1])) : kNegBig;
      }
      // ---- online softmax over this page (heads 2t, 2t+1) -------------------
      // The running max m only has to bound the logits: it moves (a warp-wide
      // max and a rescale of l and acc) only when some logit of the warp lies
      // more than kLazyMax above it, so p = 2^(lg - m) <= 2^kLazyMax and
      // P' = p n_v / sqrt(d) stays finite in fp16 for every fp16 norm n_v.
      if (__any_sync(0xffffffffu, fmaxf(lg[0], lg[2]) > m_run[0] + kLazyMax ||
                                      fmaxf(lg[1], lg[3]) > m_run[1] + kLazyMax)) {
        float alpha[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float mx = fmaxf(lg[c], lg[c + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[c], mx);
          alpha[c] = fast_exp2(m_run[c] - m_new);
          l_run[c] *= alpha[c];
          m_run[c] = m_new;
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          acc[mt][0] *= alpha[0];
          acc[mt][2] *= alpha[0];
          acc[mt][1] *= alpha[1];
          acc[mt][3] *= alpha[1];
        }
      }
      float pr[4];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        pr[c] = fast_exp2(lg[c] - m_run[c]);
        pr[c + 2] = fast_exp2(lg[c + 2] - m_run[c]);
        l_run[c] += pr[c] + pr[c + 2];
      }
      // ---- P' = p * nv / sqrt(d), transposed in registers ----------------------
      // the accumulator layout holds (token g | g + 8, heads 2t, 2t + 1); the B
      // operand wants (tokens 2t, 2t + 1 | 2t + 8, 2t + 9, head g): one 8x8 fp16
      // transpose per token half
      uint32_t pb0, pb1;
      {
        const float wg = vg ? __half2float(nv[g]) * kInvSqrtD : 0.0f;
        const float wg8 = vg8 ? __half2float(nv[g + 8]) * kInvSqrtD : 0.0f;
        pb0 = transpose8x8(pack_rn(pr[0] * wg, pr[1] * wg));
        pb1 = transpose8x8(pack_rn(pr[2] * wg8, pr[3] * wg8));
      }
      // ---- O^T += V^^T P'^T ---------------------------------------------------
      {
        const uint32_t* r0 = reinterpret_cast<const uint32_t*>(vb + (2 * t) * Gm::CBV);
        const uint32_t* r1 = reinterpret_cast<const uint32_t*>(vb + (2 * t + 1) * Gm::CBV);
        const uint32_t* r8 = reinterpret_cast<const uint32_t*>(vb + (2 * t + 8) * Gm::CBV);
        const uint32_t* r9 = reinterpret_cast<const uint32_t*>(vb + (2 * t + 9) * Gm::CBV);
        uint32_t hl0, hh0, hl1, hh1, ll0, lh0, ll1, lh1;   // [group][token pair]
        v_pairs<VBH>(v_word<VBH>(r0, g), v_word<VBH>(r1, g), hl0, hh0);
        v_pairs<VBH>(v_word<VBH>(r8, g), v_word<VBH>(r9, g), hl1, hh1);
        v_pairs<VBL>(v_word<VBL>(r0 + 2 * VBH, g), v_word<VBL>(r1 + 2 * VBH, g), ll0, lh0);
        v_pairs<VBL>(v_word<VBL>(r8 + 2 * VBH, g), v_word<VBL>(r9 + 2 * VBH, g), ll1, lh1);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const uint32_t sel = 0x7604u | (static_cast<uint32_t>(mt & 3) << 4);
          const uint32_t a0 = lds_at<0>(prmt(mt < 4 ? hl0 : hh0, lbv0, sel));
          const uint32_t a1 = lds_at<OFF1>(prmt(mt < 4 ? ll0 : lh0, lbv1, sel));
          const uint32_t a2 = lds_at<0>(prmt(mt < 4 ? hl1 : hh1, lbv0, sel));
          const uint32_t a3 = lds_at<OFF1>(prmt(mt < 4 ? ll1 : lh1, lbv1, sel));
          mma16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) issue(s);
    __syncwarp();
  }

  if (failed && lane == 0) {
    // slots i .. i+S-1 hold fills not consumed yet (slot i already gave up
    // after a timeout): let their copies land before the CTA can exit
    for (int k = drain_from; k < S; ++k) (void)mbar_wait(smem_u32(&bars[(i + k) % S]), ((i + k) / S) & 1);
  }
  // the last warp to finish resets the work counter for the next launch
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    const int total_warps = gridDim.x * W;
    if (atomicAdd(a.sched + 1, 1) == total_warps - 1) {
      a.sched[0] = 0;
      a.sched[1] = 0;
      __threadfence();
    }
  }
}

template <int W, int KBH, int KBL, int VBH, int VBL, bool QJL, bool CAUSAL = false>
cudaError_t launch_lut(const DecodeArgs& a, int items, int grid, cudaStream_t s) {
  using Gm = Geo<W, KBH, KBL, VBH, VBL, QJL>;
  static std::atomic<unsigned long long> configured{0};
  const cudaError_t e =
      smem_attr_once(lut_partials_kernel<W, KBH, KBL, VBH, VBL, QJL, CAUSAL>, Gm::SMEM, configured);
  if (e != cudaSuccess) return e;
  return launch_pdl(lut_partials_kernel<W, KBH, KBL, VBH, VBL, QJL, CAUSAL>, dim3(grid), dim3(32 * W),
                    static_cast<size_t>(Gm::SMEM), s, a, items);
}

template <int KBH, int KBL, int VBH, int VBL>
cudaError_t launch_lut_q(const DecodeArgs& a, int items, cudaStream_t s) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one CTA per SM (fewer when there are fewer chunks than SMs, or when the
  // caller caps the CTAs): a warp without a chunk exits at once, and every
  // SM's copy engines are in use
  const int cap = a.max_ctas > 0 && a.max_ctas < sms ? a.max_ctas : sms;
  const int grid = items < cap ? (items > 0 ? items : 1) : cap;
  if (a.T > 0)                         // causal (many new tokens): 16 warps
    return a.kl.qjl ? launch_lut<16, KBH, KBL, VBH, VBL, true, true>(a, items, grid, s)
                    : launch_lut<16, KBH, KBL, VBH, VBL, false, true>(a, items, grid, s);
  if (lut_warps_for(items, cap) == 12)
    return a.kl.qjl ? launch_lut<12, KBH, KBL, VBH, VBL, true>(a, items, grid, s)
                    : launch_lut<12, KBH, KBL, VBH, VBL, false>(a, items, grid, s);
  return a.kl.qjl ? launch_lut<16, KBH, KBL, VBH, VBL, true>(a, items, grid, s)
                  : launch_lut<16, KBH, KBL, VBH, VBL, false>(a, items, grid, s);
}

int combo_code(const KindLayout& kl, const KindLayout& vl) {
  return kl.g[0].bits * 1000 + kl.g[1].bits * 100 + vl.g[0].bits * 10 + vl.g[1].bits;
}

}  // namespace

int lut_decode_ctas(const KindLayout& kl, const KindLayout& vl, int m, int G) {
  if (m != 128 || kl.split != 64 || vl.split != 64 || G > 8) return 0;
  switch (combo_code(kl, vl)) {
    case 3333: case 4343: case 3232: case 4444: case 2222: case 4422: break;
    default: return 0;
  }
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

long long lut_cost(long long items, int ctas, int warps, long long chunk_cost) {
  const long long slots = static_cast<long long>(ctas > 0 ? ctas : 1) * warps;
  return (items + slots - 1) / slots * chunk_cost * warps;
}

int lut_warps_for(long long items, int ctas) {
  return lut_cost(items, ctas, 12, 1) < lut_cost(items, ctas, 16, 1) ? 12 : 16;
}

bool launch_partials_lut(const DecodeArgs& a, cudaStream_t s, cudaError_t* err) {
  if (!lut_decode_ctas(a.kl, a.vl, a.m, a.G) || !a.sched || !a.qfrag) return false;
  if ((reinterpret_cast<uintptr_t>(a.kc) | reinterpret_cast<uintptr_t>(a.vc)) & 15) return false;
  if ((a.k_page_bytes | a.v_page_bytes) & 15) return false;
  const long long items = static_cast<long long>(a.B) * a.H * a.nchunks * (a.T > 0 ? a.nqb : 1);
  if (items > (1LL << 30)) return false;
  const int n = static_cast<int>(items);
  switch (combo_code(a.kl, a.vl)) {
    case 3333: *err = launch_lut_q<3, 3, 3, 3>(a, n, s); return true;
    case 4343: *err = launch_lut_q<4, 3, 4, 3>(a, n, s); return true;
    case 3232: *err = launch_lut_q<3, 2, 3, 2>(a, n, s); return true;
    case 4444: *err = launch_lut_q<4, 4, 4, 4>(a, n, s); return true;
    case 2222: *err = launch_lut_q<2, 2, 2, 2>(a, n, s); return true;
    case 4422: *err = launch_lut_q<4, 4, 2, 2>(a, n, s); return true;
    default: return false;
  }
}

}  // namespace tq
