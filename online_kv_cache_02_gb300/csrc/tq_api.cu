// C ABI entry points: context creation, argument checks, launches, status.
#include "tq_internal.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

using namespace tq;

namespace {

// The last CUDA error a call on this host thread met (name and message).
thread_local char g_last_cuda_error[160] = "none";

tq_status cuda_fail(cudaError_t e) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return TQ_ERR_CUDA;
}

tq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TQ_OK : cuda_fail(e); }

bool valid_bits(int b) { return b >= 1 && b <= 4; }

tq_status check_config(const tq_config* c) {
  if (!c) return TQ_ERR_INVALID_ARG;
  if (c->d < 32 || c->d > kDMax || c->d % 32 || c->page_size != kPage) return TQ_ERR_UNSUPPORTED;
  if (c->m < 32 || c->m > kMaxM || c->m % 32) return TQ_ERR_INVALID_ARG;
  if (!valid_bits(c->k_bits_hi) || !valid_bits(c->k_bits_lo) || !valid_bits(c->v_bits_hi) ||
      !valid_bits(c->v_bits_lo))
    return TQ_ERR_INVALID_ARG;
  if (c->k_split < 0 || c->k_split > c->d || c->k_split % 32) return TQ_ERR_INVALID_ARG;
  if (c->v_split < 0 || c->v_split > c->d || c->v_split % 32) return TQ_ERR_INVALID_ARG;
  if (c->k_qjl != 0 && c->k_qjl != 1) return TQ_ERR_INVALID_ARG;
  if (c->codebook != TQ_CODEBOOK_GAUSSIAN && c->codebook != TQ_CODEBOOK_SPHERE) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

void fill_group(GroupBook& g, int bits, int density, int d) {
  double c[256], t[256];
  if (density == TQ_CODEBOOK_SPHERE)
    codebook_fill_sphere(bits, d, c, t);
  else
    codebook_fill(bits, c, t);
  g.bits = bits;
  g.nb = (1 << bits) - 1;
  for (int k = 0; k < 16; ++k) {
    bool in_c = k < (1 << bits), in_t = k < g.nb;
    g.c64[k] = in_c ? c[k] : 0.0;
    g.c[k] = static_cast<float>(g.c64[k]);
    g.c_lo[k] = static_cast<float>(g.c64[k] - static_cast<double>(g.c[k]));
    g.t64[k] = in_t ? t[k] : INFINITY;
    g.t[k] = in_t ? static_cast<float>(t[k]) : INFINITY;
  }
}

void fill_layout(KindLayout& L, int bits_hi, int bits_lo, int split, int d, int m, bool key, bool qjl,
                 int density) {
  fill_group(L.g[0], bits_hi, density, d);
  fill_group(L.g[1], bits_lo, density, d);
  L.split = split;
  L.code_bytes = (split * bits_hi + (d - split) * bits_lo) / 8;
  L.qjl = (key && qjl) ? 1 : 0;
  int sign_bytes = L.qjl ? m / 8 : 0;
  L.off_signs = kPage * L.code_bytes;
  L.off_norm = L.off_signs + kPage * sign_bytes;
  L.off_rnorm = L.off_norm + kPage * 2;
  L.block_bytes = L.off_norm + kPage * 2 + (L.qjl ? kPage * 2 : 0);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Element offset (in halves) of (row n, channel k) of a K-major operand tile of
// `rows` rows x 128 channels in the 128-byte-swizzled layout.
size_t swz(int n, int k, int rows) {
  const int kb = k >> 6, kk = k & 63;
  const int chunk = (kk >> 3) ^ (n & 7);
  return static_cast<size_t>(kb) * rows * 64 + static_cast<size_t>(n) * 64 + chunk * 8 + (kk & 7);
}

uint16_t to_f16(float x) {
  // round to nearest even fp16 (host); values here are |x| < 2^15 and far from subnormal issues
  uint32_t b;
  std::memcpy(&b, &x, 4);
  const uint32_t sign = (b >> 16) & 0x8000u;
  const int exp = static_cast<int>((b >> 23) & 0xFF) - 127;
  uint32_t man = b & 0x7FFFFFu;
  if (exp < -24) return static_cast<uint16_t>(sign);
  if (exp < -14) {                       // subnormal fp16
    man |= 0x800000u;
    const int shift = -exp - 14 + 13;
    uint32_t h = man >> shift;
    const uint32_t rem = man & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (h & 1u))) ++h;
    return static_cast<uint16_t>(sign | h);
  }
  uint32_t h = (static_cast<uint32_t>(exp + 15) << 10) | (man >> 13);
  const uint32_t rem = man & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) ++h;
  return static_cast<uint16_t>(sign | h);
}

float from_f16(uint16_t h) {
  const uint32_t sign = (h & 0x8000u) << 16;
  const int exp = (h >> 10) & 0x1F;
  const uint32_t man = h & 0x3FFu;
  float v;
  if (exp == 0) v = std::ldexp(static_cast<float>(man), -24);
  else v = std::ldexp(static_cast<float>(man | 0x400u), exp - 25);
  uint32_t b;
  std::memcpy(&b, &v, 4);
  b |= sign;
  std::memcpy(&v, &b, 4);
  return v;
}

// Split-K chunk length: the partials kernel keeps 3 CTAs resident per SM, so
// pick the chunk count whose CTA total fills whole waves of 3 x SMs best
// (chunks of at least 512 tokens, in multiples of 64).
int pick_chunk(int units, int max_seq_len) {
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  const long long slots = 3LL * sms;
  int best_chunk = ((max_seq_len + 63) / 64) * 64;
  if (best_chunk < 64) best_chunk = 64;
  double best_eff = -1.0;
  for (int nch = 1; nch <= 256; ++nch) {
    long long chunk = (max_seq_len + nch - 1) / nch;
    chunk = ((chunk + 63) / 64) * 64;
    if (chunk < 64) chunk = 64;
    if (chunk < 512 && nch > 1) break;
    const long long real = (max_seq_len + chunk - 1) / chunk;
    const long long ctas = real * units;
    const long long waves = (ctas + slots - 1) / slots;
    const double eff = static_cast<double>(ctas) / static_cast<double>(waves * slots);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best_chunk = static_cast<int>(chunk);
    }
  }
  return best_chunk;
}

// Chunk for the persistent kernel (one warp per chunk, chunks taken from a
// counter, ctas x 12 or 16 warp slots): the busiest warp handles
// ceil(items / slots) chunks; minimise lut_cost, that times (chunk + a
// per-chunk cost of about 32 tokens) times the warps per CTA (a warp's speed
// scales as their inverse), over both warp counts, chunks of >= 256 tokens.  items = H * sum_b ceil(L_b / chunk), estimated from the total length
// (each sequence adds half a chunk of rounding), at most every sequence full.
int pick_chunk_total(int batch, int H, long long total_tokens, int max_seq_len, int ctas) {
  long long best_cost = -1;
  int best_chunk = ((max_seq_len + kPage - 1) / kPage) * kPage;
  if (best_chunk < kPage) best_chunk = kPage;
  for (int nch = 1; nch <= 4096; ++nch) {
    long long chunk = (max_seq_len + nch - 1) / nch;
    chunk = ((chunk + kPage - 1) / kPage) * kPage;
    if (chunk < kPage) chunk = kPage;
    if (chunk < 64 && nch > 1) break;
    const long long full = static_cast<long long>(batch) * ((max_seq_len + chunk - 1) / chunk);
    const long long est = (total_tokens + chunk - 1) / chunk + batch / 2;
    const long long items = static_cast<long long>(H) * (est < full ? est : full);
    const long long cost = std::min(lut_cost(items, ctas, 12, chunk + 32), lut_cost(items, ctas, 16, chunk + 32));
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_chunk = static_cast<int>(chunk);
    }
  }
  return best_chunk;
}

// Chunk for the persistent kernel when only max_seq_len is known: every
// sequence assumed full (see pick_chunk_total, per-chunk cost 64 tokens).
int pick_chunk_warps(int units, int max_seq_len, int ctas) {
  long long best_cost = -1;
  int best_chunk = ((max_seq_len + kPage - 1) / kPage) * kPage;
  if (best_chunk < kPage) best_chunk = kPage;
  for (int nch = 1; nch <= 4096; ++nch) {
    long long chunk = (max_seq_len + nch - 1) / nch;
    chunk = ((chunk + kPage - 1) / kPage) * kPage;
    if (chunk < kPage) chunk = kPage;
    if (chunk < 64 && nch > 1) break;
    const long long real = (max_seq_len + chunk - 1) / chunk;
    const long long items = real * units;
    const long long cost = std::min(lut_cost(items, ctas, 12, chunk + 64), lut_cost(items, ctas, 16, chunk + 64));
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_chunk = static_cast<int>(chunk);
    }
  }
  return best_chunk;
}

}  // namespace

extern "C" tq_status tq_config_init(tq_config* cfg, int d, int b, int m, uint64_t seed) {
  if (!cfg) return TQ_ERR_INVALID_ARG;
  cfg->d = d;
  cfg->m = m;
  cfg->page_size = kPage;
  cfg->k_bits_hi = cfg->k_bits_lo = b;
  cfg->v_bits_hi = cfg->v_bits_lo = b;
  cfg->k_split = cfg->v_split = d / 64 * 32;          // half the channels, rounded down to a multiple of 32
  cfg->k_qjl = 1;
  cfg->seed = seed;
  cfg->codebook = TQ_CODEBOOK_GAUSSIAN;
  return check_config(cfg);
}

extern "C" tq_status tq_create(int d, int b, int m, uint64_t seed, tq_ctx** out) {
  tq_config cfg;
  tq_status st = tq_config_init(&cfg, d, b, m, seed);
  if (st != TQ_OK) return st;
  return tq_create_ex(&cfg, out);
}

extern "C" tq_status tq_create_ex(const tq_config* cfg, tq_ctx** out) {
  if (!out) return TQ_ERR_INVALID_ARG;
  *out = nullptr;
  tq_status st = check_config(cfg);
  if (st != TQ_OK) return st;
  const int d = cfg->d, m = cfg->m;
  tq_ctx* ctx = new (std::nothrow) tq_ctx();
  if (!ctx) return TQ_ERR_OOM;
  ctx->cfg = *cfg;
  if (cudaGetDevice(&ctx->device) != cudaSuccess) {
    delete ctx;
    return TQ_ERR_CUDA;
  }
  fill_layout(ctx->kl, cfg->k_bits_hi, cfg->k_bits_lo, cfg->k_split, d, m, true, cfg->k_qjl != 0, cfg->codebook);
  fill_layout(ctx->vl, cfg->v_bits_hi, cfg->v_bits_lo, cfg->v_split, d, m, false, false, cfg->codebook);

  std::vector<double> pi(static_cast<size_t>(d) * d), s(static_cast<size_t>(m) * d);
  rotation_fill(d, cfg->seed, pi.data());
  qjl_fill(m, d, cfg->seed, s.data());
  std::vector<float> pit(d * d), pif(d * d), st_(static_cast<size_t>(d) * m);
  for (int i = 0; i < d; ++i)
    for (int k = 0; k < d; ++k) {
      pif[i * d + k] = static_cast<float>(pi[i * d + k]);
      pit[k * d + i] = static_cast<float>(pi[i * d + k]);
    }
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < d; ++j) st_[static_cast<size_t>(j) * m + i] = static_cast<float>(s[i * d + j]);

  // tensor-core operand tiles (d = 128 only: the swizzled layout holds 64-channel
  // blocks) and double-float refinement tables
  std::vector<uint16_t> pih(d * d), pil(d * d), sh(static_cast<size_t>(m) * d), sl(static_cast<size_t>(m) * d);
  std::vector<float> pidf(static_cast<size_t>(d) * d * 2);
  for (int i = 0; i < d; ++i)
    for (int k = 0; k < d; ++k) {
      if (d == kD) {
        const double v = pi[i * d + k] * kPiScale;   // scaled so the low part stays a normal fp16
        const uint16_t hi = to_f16(static_cast<float>(v));
        pih[swz(i, k, d)] = hi;
        pil[swz(i, k, d)] = to_f16(static_cast<float>(v - static_cast<double>(from_f16(hi))));
      }
      const float phi = static_cast<float>(pi[i * d + k]);
      pidf[(i * d + k) * 2] = phi;
      pidf[(i * d + k) * 2 + 1] = static_cast<float>(pi[i * d + k] - static_cast<double>(phi));
    }
  if (d == kD)
    for (int p = 0; p < m; ++p)
      for (int j = 0; j < d; ++j) {
        const uint16_t hi = to_f16(static_cast<float>(s[p * d + j]));
        sh[swz(p, j, m)] = hi;
        sl[swz(p, j, m)] = to_f16(static_cast<float>(s[p * d + j] - static_cast<double>(from_f16(hi))));
      }
  std::vector<float> adf(static_cast<size_t>(m) * d * 2), sdf(static_cast<size_t>(m) * d * 2);
  std::vector<float> wt(static_cast<size_t>(d) * (d + m));   // W = [Pi; S Pi], stored transposed
  for (int r = 0; r < d; ++r)
    for (int k = 0; k < d; ++k) wt[static_cast<size_t>(k) * (d + m) + r] = static_cast<float>(pi[r * d + k]);
  for (int p = 0; p < m; ++p)
    for (int k = 0; k < d; ++k) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += s[p * d + i] * pi[i * d + k];   // (S Pi)[p][k]
      wt[static_cast<size_t>(k) * (d + m) + d + p] = static_cast<float>(acc);
      const float hi = static_cast<float>(acc);
      adf[(p * d + k) * 2] = hi;
      adf[(p * d + k) * 2 + 1] = static_cast<float>(acc - static_cast<double>(hi));
      const float shi = static_cast<float>(s[p * d + k]);
      sdf[(p * d + k) * 2] = shi;
      sdf[(p * d + k) * 2 + 1] = static_cast<float>(s[p * d + k] - static_cast<double>(shi));
    }
  size_t o_pit = 0;
  size_t o_pi = align256(o_pit + sizeof(float) * d * d);
  size_t o_pi64 = align256(o_pi + sizeof(float) * d * d);
  size_t o_st = align256(o_pi64 + sizeof(double) * d * d);
  size_t o_s64 = align256(o_st + sizeof(float) * d * m);
  size_t o_pih = align256(o_s64 + sizeof(double) * d * m);
  size_t o_pil = align256(o_pih + sizeof(uint16_t) * d * d);
  size_t o_sh = align256(o_pil + sizeof(uint16_t) * d * d);
  size_t o_sl = align256(o_sh + sizeof(uint16_t) * d * m);
  size_t o_adf = align256(o_sl + sizeof(uint16_t) * d * m);
  size_t o_sdf = align256(o_adf + sizeof(float) * d * m * 2);
  size_t o_pidf = align256(o_sdf + sizeof(float) * d * m * 2);
  size_t o_wt = align256(o_pidf + sizeof(float) * d * d * 2);
  size_t o_err = align256(o_wt + sizeof(float) * d * (d + m));
  size_t o_cnt = align256(o_err + sizeof(uint32_t));
  size_t total = align256(o_cnt + 2 * sizeof(unsigned long long));
  void* blk = nullptr;
  if (cudaMalloc(&blk, total) != cudaSuccess) {
    delete ctx;
    cudaGetLastError();
    return TQ_ERR_OOM;
  }
  char* b = static_cast<char*>(blk);
  ctx->dev_block = blk;
  ctx->tab.pit = reinterpret_cast<float*>(b + o_pit);
  ctx->tab.pi = reinterpret_cast<float*>(b + o_pi);
  ctx->tab.pi64 = reinterpret_cast<double*>(b + o_pi64);
  ctx->tab.st = reinterpret_cast<float*>(b + o_st);
  ctx->tab.s64 = reinterpret_cast<double*>(b + o_s64);
  ctx->tab.pih_sw = reinterpret_cast<unsigned short*>(b + o_pih);
  ctx->tab.pil_sw = reinterpret_cast<unsigned short*>(b + o_pil);
  ctx->tab.sh_sw = reinterpret_cast<unsigned short*>(b + o_sh);
  ctx->tab.sl_sw = reinterpret_cast<unsigned short*>(b + o_sl);
  ctx->tab.a_df = reinterpret_cast<float*>(b + o_adf);
  ctx->tab.s_df = reinterpret_cast<float*>(b + o_sdf);
  ctx->tab.pi_df = reinterpret_cast<float*>(b + o_pidf);
  ctx->tab.wt = reinterpret_cast<float*>(b + o_wt);
  ctx->tab.err = reinterpret_cast<uint32_t*>(b + o_err);
  ctx->tab.counters = reinterpret_cast<unsigned long long*>(b + o_cnt);
  bool ok = cudaMemcpy(ctx->tab.pit, pit.data(), sizeof(float) * d * d, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.pi, pif.data(), sizeof(float) * d * d, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.pi64, pi.data(), sizeof(double) * d * d, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.st, st_.data(), sizeof(float) * d * m, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.s64, s.data(), sizeof(double) * d * m, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.pih_sw, pih.data(), 2 * d * d, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.pil_sw, pil.data(), 2 * d * d, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.sh_sw, sh.data(), 2 * d * m, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.sl_sw, sl.data(), 2 * d * m, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.pi_df, pidf.data(), sizeof(float) * d * d * 2, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.a_df, adf.data(), sizeof(float) * d * m * 2, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.s_df, sdf.data(), sizeof(float) * d * m * 2, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(ctx->tab.wt, wt.data(), sizeof(float) * d * (d + m), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemset(b + o_err, 0, total - o_err) == cudaSuccess;
  if (!ok) { cudaFree(blk); delete ctx; cudaGetLastError(); return TQ_ERR_CUDA; }
  *out = ctx;
  return TQ_OK;
}

extern "C" tq_status tq_destroy(tq_ctx* ctx) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  cudaError_t e = cudaFree(ctx->dev_block);
  delete ctx;
  return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

extern "C" tq_status tq_get_config(const tq_ctx* ctx, tq_config* cfg) {
  if (!ctx || !cfg) return TQ_ERR_INVALID_ARG;
  *cfg = ctx->cfg;
  return TQ_OK;
}

extern "C" tq_status tq_cache_layout(const tq_ctx* ctx, int num_kv_heads, size_t* kpb, size_t* vpb) {
  if (!ctx || num_kv_heads < 1 || (!kpb && !vpb)) return TQ_ERR_INVALID_ARG;
  if (kpb) *kpb = static_cast<size_t>(ctx->kl.block_bytes) * num_kv_heads;
  if (vpb) *vpb = static_cast<size_t>(ctx->vl.block_bytes) * num_kv_heads;
  return TQ_OK;
}

namespace {
tq_status quantize_impl(const tq_ctx* ctx, const void* k, const void* v, tq_dtype dtype, int batch, int n_new, int H,
                        const int32_t* start_pos, const int32_t* block_table, int maxp, int num_pages, void* k_cache,
                        void* v_cache, void* stream, int max_ctas);
}  // namespace

extern "C" tq_status tq_quantize(const tq_ctx* ctx, const void* k, const void* v, tq_dtype dtype,
                                 int batch, int n_new, int H, const int32_t* start_pos,
                                 const int32_t* block_table, int maxp, int num_pages, void* k_cache,
                                 void* v_cache, void* stream) {
  return quantize_impl(ctx, k, v, dtype, batch, n_new, H, start_pos, block_table, maxp, num_pages, k_cache, v_cache,
                       stream, 0);
}

namespace {
tq_status quantize_impl(const tq_ctx* ctx, const void* k, const void* v, tq_dtype dtype, int batch, int n_new, int H,
                        const int32_t* start_pos, const int32_t* block_table, int maxp, int num_pages, void* k_cache,
                        void* v_cache, void* stream, int max_ctas) {
  if (!ctx || (!k && !v) || batch < 0 || n_new < 0 || H < 1 || maxp < 1 || num_pages < 1)
    return TQ_ERR_INVALID_ARG;
  if (dtype != TQ_BF16 && dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if ((k && !k_cache) || (v && !v_cache)) return TQ_ERR_INVALID_ARG;
  if (batch == 0 || n_new == 0) return TQ_OK;
  if (!start_pos || !block_table) return TQ_ERR_INVALID_ARG;
  if (static_cast<long long>(batch) * n_new * H > (1LL << 31) - 1) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  QuantizeArgs args[2]{};
  for (int kind = 0; kind < 2; ++kind) {
    QuantizeArgs& a = args[kind];
    a.x = kind == 0 ? k : v;
    a.f32 = dtype == TQ_F32;
    a.batch = batch;
    a.n_new = n_new;
    a.H = H;
    a.start_pos = start_pos;
    a.block_table = block_table;
    a.maxp = maxp;
    a.num_pages = num_pages;
    a.cache = static_cast<uint8_t*>(kind == 0 ? k_cache : v_cache);
    a.lay = kind == 0 ? ctx->kl : ctx->vl;
    a.page_bytes = static_cast<long long>(a.lay.block_bytes) * H;
    a.m = ctx->cfg.m;
    a.tab = ctx->tab;
    a.max_ctas = max_ctas;
  }
  cudaError_t e = cudaSuccess;
  if (ctx->cfg.d != kD) {                 // head dimensions other than 128: CUDA-core kernel
    for (int kind = 0; kind < 2; ++kind) {
      if (!args[kind].x) continue;
      const cudaError_t eg = launch_quantize_generic(args[kind], ctx->cfg.d, s);
      if (eg != cudaSuccess) return cuda_fail(eg);
    }
    return TQ_OK;
  }
  if (launch_quantize_pipe(args[0], args[1], s, &e)) return cuda_status(e);
  if (launch_quantize_tc(args[0], args[1], s, &e)) return cuda_status(e);
  for (int kind = 0; kind < 2; ++kind) {
    if (!args[kind].x) continue;
    const cudaError_t ek = launch_quantize(args[kind], s);
    if (ek != cudaSuccess) return cuda_fail(ek);
  }
  return TQ_OK;
}
}  // namespace

namespace {
int nchunks_for(int max_seq_len, int chunk) { return max_seq_len <= 0 ? 1 : (max_seq_len + chunk - 1) / chunk; }

// Causal attention on the tensor cores: fp16 query words (48 x 16 B per block
// row), partials (130 floats per block row and chunk), the work counters.
size_t causal_tc_ws_bytes(long long nblk, int nch) {
  return align256(static_cast<size_t>(nblk) * 128 * 48 * 16) +
         align256(static_cast<size_t>(nblk) * nch * (kD + 2) * 128 * sizeof(float)) + 256;
}

size_t ws_bytes(int B, int Hq, int d, int m, int nch) {
  return align256(sizeof(float) * static_cast<size_t>(B) * Hq * (d + m)) +
         align256(sizeof(float) * static_cast<size_t>(B) * Hq * nch * (d + 2)) +
         align256(sizeof(uint32_t) * static_cast<size_t>(B) * Hq * kQFragWords) + 256;   // + query fragments, work counters
}
}  // namespace

extern "C" tq_status tq_workspace_size(const tq_ctx* ctx, int batch, int Hq, int max_seq_len,
                                       int chunk_tokens, size_t* bytes) {
  if (!ctx || !bytes || batch < 0 || Hq < 1 || max_seq_len < 0 || chunk_tokens < 0 ||
      chunk_tokens % kPage)
    return TQ_ERR_INVALID_ARG;
  int chunk = chunk_tokens ? chunk_tokens : 0;
  if (!chunk) {
    // the automatic chunk depends on the KV-head count, which is not known
    // here; size for the smallest chunk the automatic choice can pick
    chunk = 64;
  }
  *bytes = ws_bytes(batch, Hq, ctx->cfg.d, ctx->cfg.m, nchunks_for(max_seq_len, chunk));
  return TQ_OK;
}

namespace {
int sm_count() {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

}  // namespace

extern "C" tq_status tq_decode_chunk(const tq_ctx* ctx, int batch, int Hq, int H, long long total_tokens,
                                     int max_seq_len, int fused_append, int* chunk_tokens) {
  if (!ctx || !chunk_tokens || batch < 1 || Hq < 1 || H < 1 || Hq % H || max_seq_len < 0 || total_tokens < 0 ||
      total_tokens > static_cast<long long>(batch) * max_seq_len)
    return TQ_ERR_INVALID_ARG;
  (void)fused_append;   // the fused step's partials kernel has every SM (the append runs before it)
  const int ctas = ctx->cfg.d == kD ? lut_decode_ctas(ctx->kl, ctx->vl, ctx->cfg.m, Hq / H) : 0;
  if (ctas > 0)
    *chunk_tokens = pick_chunk_total(batch, H, total_tokens, max_seq_len, ctas);
  else
    *chunk_tokens = pick_chunk(batch * H, max_seq_len);
  return TQ_OK;
}

extern "C" tq_status tq_decode_attention(const tq_ctx* ctx, const void* q, tq_dtype dtype, int batch,
                                         int Hq, int H, const int32_t* seq_lens, int max_seq_len,
                                         const int32_t* block_table, int maxp, int num_pages,
                                         const void* k_cache, const void* v_cache, int chunk_tokens,
                                         float softmax_scale, float* out, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  return tq_decode_attention_ex(ctx, q, dtype, batch, Hq, H, seq_lens, max_seq_len, block_table, maxp, num_pages,
                                k_cache, v_cache, chunk_tokens, softmax_scale, out, workspace, workspace_bytes,
                                TQ_STAGE_ALL, stream);
}

namespace {
// The fused decode step (tq_append_decode): the append kernel, then qprep as
// its dependent launch (overlapping it, finishing after it), the partials
// kernel over the L + 1 tokens and the merge.  Optional events bracket the
// partials launch.
struct FusedStep {
  cudaEvent_t partials_begin, partials_end;
};

// The tensor-core decode multiplies fp16 operands (q~, u, centroids): its logit
// error grows with |softmax_scale|, and the 2e-3 output bar holds up to
// 1/sqrt(d).  Larger scales run the fp32 CUDA-core kernels.
bool precise_scale(const tq_ctx* ctx, float softmax_scale) {
  return std::fabs(static_cast<double>(softmax_scale)) > (1.0 + 1e-6) / std::sqrt(static_cast<double>(ctx->cfg.d));
}

tq_status decode_impl(const tq_ctx* ctx, const void* q, tq_dtype dtype, int batch, int Hq, int H,
                      const int32_t* seq_lens, int len_add, int max_seq_len, const int32_t* block_table, int maxp,
                      int num_pages, const void* k_cache, const void* v_cache, int chunk_tokens,
                      float softmax_scale, float* out, void* workspace, size_t workspace_bytes, int stages,
                      void* stream, const FusedStep* fused = nullptr) {
  if (stages < 1 || stages > TQ_STAGE_ALL) return TQ_ERR_INVALID_ARG;
  if (!ctx || batch < 0 || Hq < 1 || H < 1 || Hq % H || max_seq_len < 0 || maxp < 1 ||
      num_pages < 1 || chunk_tokens < 0 || chunk_tokens % kPage)
    return TQ_ERR_INVALID_ARG;
  if (dtype != TQ_BF16 && dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return TQ_ERR_INVALID_ARG;
  if (Hq / H > kMaxGroup) return TQ_ERR_UNSUPPORTED;
  if (batch == 0) return TQ_OK;
  if (!q || !seq_lens || !block_table || !k_cache || !v_cache || !out || !workspace)
    return TQ_ERR_INVALID_ARG;
  const bool generic = ctx->cfg.d != kD || precise_scale(ctx, softmax_scale);
  int lut_ctas = generic ? 0 : lut_decode_ctas(ctx->kl, ctx->vl, ctx->cfg.m, Hq / H);
  int chunk = chunk_tokens              ? chunk_tokens
              : lut_ctas > 0            ? pick_chunk_warps(batch * H, max_seq_len, lut_ctas)
                                        : pick_chunk(batch * H, max_seq_len);
  int nch = nchunks_for(max_seq_len, chunk);
  const int d = ctx->cfg.d, m = ctx->cfg.m;
  size_t need = ws_bytes(batch, Hq, d, m, nch);
  if (workspace_bytes < need) return TQ_ERR_WORKSPACE;
  if (static_cast<long long>(nch) > 65535 || H > 65535 || batch > 65535) return TQ_ERR_UNSUPPORTED;
  DecodeArgs a{};
  a.q = q;
  a.f32 = dtype == TQ_F32;
  a.B = batch;
  a.Hq = Hq;
  a.H = H;
  a.G = Hq / H;
  a.seq_lens = seq_lens;
  a.len_add = len_add;
  a.max_seq_len = max_seq_len;
  a.block_table = block_table;
  a.maxp = maxp;
  a.num_pages = num_pages;
  a.kc = static_cast<const uint8_t*>(k_cache);
  a.vc = static_cast<const uint8_t*>(v_cache);
  a.kl = ctx->kl;
  a.vl = ctx->vl;
  a.k_page_bytes = static_cast<long long>(ctx->kl.block_bytes) * H;
  a.v_page_bytes = static_cast<long long>(ctx->vl.block_bytes) * H;
  a.chunk = chunk;
  a.nchunks = nch;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.m = m;
  a.tab = ctx->tab;
  char* w = static_cast<char*>(workspace);
  a.qprep = reinterpret_cast<float*>(w);
  a.part = reinterpret_cast<float*>(w + align256(sizeof(float) * static_cast<size_t>(batch) * Hq * (d + m)));
  const size_t o_frag = align256(sizeof(float) * static_cast<size_t>(batch) * Hq * (d + m)) +
                        align256(sizeof(float) * static_cast<size_t>(batch) * Hq * nch * (d + 2));
  a.qfrag = reinterpret_cast<uint32_t*>(w + o_frag);
  a.sched = reinterpret_cast<int*>(w + o_frag + align256(sizeof(uint32_t) * static_cast<size_t>(batch) * Hq * kQFragWords));
  a.out = out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (generic) return cuda_status(launch_decode_generic(a, d, stages, st));
  if (!fused) return cuda_status(launch_decode(a, stages, st));
  a.chained = 1;
  bool ok = launch_decode(a, TQ_STAGE_QPREP, st) == cudaSuccess;
  if (ok && fused->partials_begin) ok = cudaEventRecord(fused->partials_begin, st) == cudaSuccess;
  ok = ok && launch_decode(a, TQ_STAGE_PARTIALS, st) == cudaSuccess;
  if (ok && fused->partials_end) ok = cudaEventRecord(fused->partials_end, st) == cudaSuccess;
  ok = ok && launch_decode(a, TQ_STAGE_MERGE, st) == cudaSuccess;
  return ok ? TQ_OK : cuda_fail(cudaGetLastError());
}
}  // namespace

extern "C" tq_status tq_decode_attention_ex(const tq_ctx* ctx, const void* q, tq_dtype dtype, int batch,
                                            int Hq, int H, const int32_t* seq_lens, int max_seq_len,
                                            const int32_t* block_table, int maxp, int num_pages,
                                            const void* k_cache, const void* v_cache, int chunk_tokens,
                                            float softmax_scale, float* out, void* workspace,
                                            size_t workspace_bytes, int stages, void* stream) {
  return decode_impl(ctx, q, dtype, batch, Hq, H, seq_lens, 0, max_seq_len, block_table, maxp, num_pages, k_cache,
                     v_cache, chunk_tokens, softmax_scale, out, workspace, workspace_bytes, stages, stream);
}

extern "C" tq_status tq_append_decode(const tq_ctx* ctx, const void* k_new, const void* v_new, const void* q,
                                      tq_dtype dtype, int batch, int Hq, int H, const int32_t* seq_lens,
                                      int max_seq_len, const int32_t* block_table, int maxp, int num_pages,
                                      void* k_cache, void* v_cache, int chunk_tokens, float softmax_scale,
                                      float* out, void* workspace, size_t workspace_bytes, void* stream) {
  return tq_append_decode_ex(ctx, k_new, v_new, q, dtype, batch, Hq, H, seq_lens, max_seq_len, block_table, maxp,
                             num_pages, k_cache, v_cache, chunk_tokens, softmax_scale, out, workspace,
                             workspace_bytes, stream, nullptr, nullptr);
}

extern "C" tq_status tq_append_decode_ex(const tq_ctx* ctx, const void* k_new, const void* v_new, const void* q,
                                         tq_dtype dtype, int batch, int Hq, int H, const int32_t* seq_lens,
                                         int max_seq_len, const int32_t* block_table, int maxp, int num_pages,
                                         void* k_cache, void* v_cache, int chunk_tokens, float softmax_scale,
                                         float* out, void* workspace, size_t workspace_bytes, void* stream,
                                         void* partials_begin, void* partials_end) {
  if (!ctx || !k_new || !v_new || batch < 0 || H < 1 || Hq < 1 || Hq % H || max_seq_len < 1)
    return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  // check the decode arguments before anything is launched
  size_t need = 0;
  tq_status st = tq_workspace_size(ctx, batch, Hq, max_seq_len, chunk_tokens, &need);
  if (st != TQ_OK) return st;
  if (!q || !out || !workspace || !seq_lens || !block_table) return TQ_ERR_INVALID_ARG;
  if (Hq / H > kMaxGroup) return TQ_ERR_UNSUPPORTED;
  if (dtype != TQ_BF16 && dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || maxp < 1 || num_pages < 1) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return TQ_ERR_INVALID_ARG;
  if (static_cast<long long>(batch) * H > (1LL << 31) - 1) return TQ_ERR_INVALID_ARG;
  if (ctx->cfg.d != kD || precise_scale(ctx, softmax_scale)) {   // CUDA-core decode: append, then decode L + 1
    st = quantize_impl(ctx, k_new, v_new, dtype, batch, 1, H, seq_lens, block_table, maxp, num_pages, k_cache, v_cache,
                       stream, 0);
    if (st != TQ_OK) return st;
    if (partials_begin && cudaEventRecord(static_cast<cudaEvent_t>(partials_begin), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return cuda_fail(cudaGetLastError());
    st = decode_impl(ctx, q, dtype, batch, Hq, H, seq_lens, 1, max_seq_len, block_table, maxp, num_pages, k_cache,
                     v_cache, chunk_tokens, softmax_scale, out, workspace, workspace_bytes, TQ_STAGE_ALL, stream);
    if (st == TQ_OK && partials_end &&
        cudaEventRecord(static_cast<cudaEvent_t>(partials_end), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return cuda_fail(cudaGetLastError());
    return st;
  }
  // one stream: the append kernel (a warp per new vector), then the decode
  // over L + 1 tokens with qprep launched dependent on the append
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  QuantizeArgs qa[2]{};
  for (int kind = 0; kind < 2; ++kind) {
    QuantizeArgs& x = qa[kind];
    x.x = kind == 0 ? k_new : v_new;
    x.f32 = dtype == TQ_F32;
    x.batch = batch;
    x.n_new = 1;
    x.H = H;
    x.start_pos = seq_lens;
    x.block_table = block_table;
    x.maxp = maxp;
    x.num_pages = num_pages;
    x.cache = static_cast<uint8_t*>(kind == 0 ? k_cache : v_cache);
    x.lay = kind == 0 ? ctx->kl : ctx->vl;
    x.page_bytes = static_cast<long long>(x.lay.block_bytes) * H;
    x.m = ctx->cfg.m;
    x.tab = ctx->tab;
  }
  cudaError_t e = cudaSuccess;
  if (!launch_append(qa[0], qa[1], s, &e)) {
    st = quantize_impl(ctx, k_new, v_new, dtype, batch, 1, H, seq_lens, block_table, maxp, num_pages, k_cache,
                       v_cache, stream, 0);
    if (st != TQ_OK) return st;
  } else if (e != cudaSuccess) {
    return cuda_fail(e);
  }
  FusedStep f{static_cast<cudaEvent_t>(partials_begin), static_cast<cudaEvent_t>(partials_end)};
  return decode_impl(ctx, q, dtype, batch, Hq, H, seq_lens, 1, max_seq_len, block_table, maxp, num_pages, k_cache,
                     v_cache, chunk_tokens, softmax_scale, out, workspace, workspace_bytes, TQ_STAGE_ALL, stream, &f);
}

// ---------------------------------------------------------------------------
// multi-query causal attention (many new tokens per sequence)
// ---------------------------------------------------------------------------
extern "C" tq_status tq_causal_workspace_size(const tq_ctx* ctx, int batch, int n_new, int Hq, int max_seq_len,
                                              int chunk_tokens, size_t* bytes) {
  if (!ctx || !bytes || batch < 0 || n_new < 1 || Hq < 1 || max_seq_len < n_new || chunk_tokens < 0 ||
      chunk_tokens % kPage)
    return TQ_ERR_INVALID_ARG;
  if (causal_tc_supported(ctx->kl, ctx->vl, ctx->cfg.m) && chunk_tokens <= causal_tc_max_chunk()) {
    // tensor-core path: at most Hq ceil(n_new / 128) query blocks per sequence, chunks of at least 256
    const long long nblk = static_cast<long long>(batch) * Hq * ((n_new + 127) / 128);
    *bytes = causal_tc_ws_bytes(nblk, nchunks_for(max_seq_len, chunk_tokens ? chunk_tokens : 256));
    return TQ_OK;
  }
  const int chunk = chunk_tokens ? chunk_tokens : 64;   // the smallest automatic chunk
  *bytes = ws_bytes(static_cast<int>(static_cast<long long>(batch) * n_new), Hq, ctx->cfg.d, ctx->cfg.m,
                    nchunks_for(max_seq_len, chunk));
  return TQ_OK;
}

extern "C" tq_status tq_causal_attention(const tq_ctx* ctx, const void* q, tq_dtype dtype, int batch, int n_new,
                                         int Hq, int H, const int32_t* start_pos, int max_seq_len,
                                         const int32_t* block_table, int maxp, int num_pages, const void* k_cache,
                                         const void* v_cache, int chunk_tokens, float softmax_scale, float* out,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!ctx || batch < 0 || n_new < 1 || Hq < 1 || H < 1 || Hq % H || max_seq_len < n_new || maxp < 1 ||
      num_pages < 1 || chunk_tokens < 0 || chunk_tokens % kPage)
    return TQ_ERR_INVALID_ARG;
  if (dtype != TQ_BF16 && dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return TQ_ERR_INVALID_ARG;
  if (Hq / H > kMaxGroup || ctx->cfg.d != kD || precise_scale(ctx, softmax_scale)) return TQ_ERR_UNSUPPORTED;
  const int lut_ctas = lut_decode_ctas(ctx->kl, ctx->vl, ctx->cfg.m, Hq / H);
  if (lut_ctas <= 0) return TQ_ERR_UNSUPPORTED;        // the bit widths the persistent kernel takes
  if (batch == 0) return TQ_OK;
  if (!q || !start_pos || !block_table || !k_cache || !v_cache || !out || !workspace) return TQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15) return TQ_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(batch) * n_new;
  if (rows * Hq > (1LL << 31) - 1 || rows > 65535LL * 65535LL) return TQ_ERR_UNSUPPORTED;
  const int G = Hq / H;
  // tensor cores: blocks of 128 query rows, chunks of at most 1024 tokens;
  // else the lookup-table partials kernel's causal instances (8 rows a block)
  const bool tc = causal_tc_supported(ctx->kl, ctx->vl, ctx->cfg.m) && chunk_tokens <= causal_tc_max_chunk();
  const int rows_blk = tc ? causal_tc_block_rows() : 8;
  const int nqb = static_cast<int>((static_cast<long long>(n_new) * G + rows_blk - 1) / rows_blk);
  int chunk = chunk_tokens;
  if (!chunk && tc) {                 // the largest chunk that still gives three items per SM
    const long long bhq = static_cast<long long>(batch) * H * nqb;
    chunk = causal_tc_max_chunk();
    while (chunk > 256 && bhq * nchunks_for(max_seq_len, chunk) < 3LL * sm_count()) chunk /= 2;
  } else if (!chunk) {
    chunk = pick_chunk_warps(static_cast<int>(std::min<long long>(static_cast<long long>(batch) * H * nqb, 1 << 30)),
                             max_seq_len, lut_ctas);
  }
  const int nch = nchunks_for(max_seq_len, chunk);
  const int d = ctx->cfg.d, m = ctx->cfg.m;
  const long long nblk = static_cast<long long>(batch) * H * nqb;
  if (workspace_bytes < (tc ? causal_tc_ws_bytes(nblk, nch) : ws_bytes(static_cast<int>(rows), Hq, d, m, nch)))
    return TQ_ERR_WORKSPACE;
  if (static_cast<long long>(batch) * H * nqb * nch > (1LL << 30) || nch > 65535) return TQ_ERR_UNSUPPORTED;
  DecodeArgs a{};
  a.q = q;
  a.f32 = dtype == TQ_F32;
  a.B = batch;
  a.Hq = Hq;
  a.H = H;
  a.G = G;
  a.seq_lens = start_pos;
  a.len_add = n_new;
  a.max_seq_len = max_seq_len;
  a.block_table = block_table;
  a.maxp = maxp;
  a.num_pages = num_pages;
  a.kc = static_cast<const uint8_t*>(k_cache);
  a.vc = static_cast<const uint8_t*>(v_cache);
  a.kl = ctx->kl;
  a.vl = ctx->vl;
  a.k_page_bytes = static_cast<long long>(ctx->kl.block_bytes) * H;
  a.v_page_bytes = static_cast<long long>(ctx->vl.block_bytes) * H;
  a.chunk = chunk;
  a.nchunks = nch;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.m = m;
  a.tab = ctx->tab;
  a.T = n_new;
  a.nqb = nqb;
  char* w = static_cast<char*>(workspace);
  const size_t o_part = align256(sizeof(float) * static_cast<size_t>(rows) * Hq * (d + m));
  const size_t o_frag = o_part + align256(sizeof(float) * static_cast<size_t>(rows) * Hq * nch * (d + 2));
  a.qprep = reinterpret_cast<float*>(w);
  a.part = reinterpret_cast<float*>(w + o_part);
  a.qfrag = reinterpret_cast<uint32_t*>(w + o_frag);
  a.sched = reinterpret_cast<int*>(w + o_frag + align256(sizeof(uint32_t) * static_cast<size_t>(rows) * Hq * kQFragWords));
  a.out = out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!tc) return cuda_status(launch_decode(a, TQ_STAGE_ALL, st));
  a.qfrag = nullptr;
  a.qhalf = 1;                        // fp16 query words and partials stored by query block
  a.qprep = reinterpret_cast<float*>(w);
  a.part = reinterpret_cast<float*>(w + align256(static_cast<size_t>(nblk) * 128 * 48 * 16));
  a.sched = reinterpret_cast<int*>(reinterpret_cast<char*>(a.part) +
                                   align256(static_cast<size_t>(nblk) * nch * (kD + 2) * 128 * sizeof(float)));
  cudaError_t e = launch_decode(a, TQ_STAGE_QPREP, st);
  if (e == cudaSuccess) e = launch_causal_tc(a, nqb, st);
  if (e == cudaSuccess) e = launch_decode(a, TQ_STAGE_MERGE, st);
  return cuda_status(e);
}

extern "C" tq_status tq_check_device_status(const tq_ctx* ctx, uint32_t* flags) {
  if (!ctx) return TQ_ERR_INVALID_ARG;
  uint32_t h = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaMemcpy(&h, ctx->tab.err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaMemset(ctx->tab.err, 0, sizeof(h)) != cudaSuccess) return TQ_ERR_CUDA;
  if (flags) *flags = h;
  return h ? TQ_ERR_DEVICE_CHECK : TQ_OK;
}

extern "C" tq_status tq_refine_counters(const tq_ctx* ctx, unsigned long long out[2], int reset) {
  if (!ctx || !out) return TQ_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaMemcpy(out, ctx->tab.counters, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TQ_ERR_CUDA;
  if (reset && cudaMemset(ctx->tab.counters, 0, 2 * sizeof(unsigned long long)) != cudaSuccess) return TQ_ERR_CUDA;
  return TQ_OK;
}

extern "C" const char* tq_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_OOM: return "out of device memory";
    case TQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case TQ_ERR_DEVICE_CHECK: return "device-side range check failed (input skipped)";
    case TQ_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

// ---------------------------------------------------------------------------
// inner-product search
// ---------------------------------------------------------------------------
namespace {
// Workspace of a search: the q~/u rows, then the tensor-core path's candidate
// lists, or the CUDA-core path's [nq][n_db] scores (k_top > 0); the rows alone
// for tq_search_scores (k_top = 0).
size_t search_bytes(const tq_ctx* ctx, int nq, int n_db, int k_top) {
  const size_t rows = search_qrows_bytes(nq, ctx->cfg.m);
  if (k_top == 0) return rows + 256;
  if (search_tc_supported(ctx->kl, ctx->cfg.m, k_top)) return rows + search_tc_cand_bytes() + 256;
  return rows + sizeof(float) * static_cast<size_t>(nq) * n_db + 256;
}

DecodeArgs search_args(const tq_ctx* ctx, const void* q, tq_dtype dtype, int nq, void* workspace) {
  DecodeArgs a{};
  a.q = q;
  a.f32 = dtype == TQ_F32 ? 1 : 0;
  a.B = 1;
  a.Hq = nq;
  a.H = 1;
  a.G = nq;
  a.m = ctx->cfg.m;
  a.kl = ctx->kl;
  a.vl = ctx->vl;
  a.tab = ctx->tab;
  a.qprep = static_cast<float*>(workspace);
  a.qfrag = nullptr;
  a.sched = nullptr;
  return a;
}

// Checks shared by tq_search and tq_search_scores, before any launch.
tq_status search_check(const tq_ctx* ctx, const void* q, tq_dtype dtype, int nq, const void* k_cache,
                       const int32_t* block_table, int num_pages, int n_db, const void* workspace) {
  if (!ctx || !q || !k_cache || !block_table || !workspace) return TQ_ERR_INVALID_ARG;
  if (dtype != TQ_BF16 && dtype != TQ_F32) return TQ_ERR_INVALID_ARG;
  if (nq < 1 || n_db < 1 || num_pages < 1) return TQ_ERR_INVALID_ARG;
  if (static_cast<long long>(num_pages) * kPage < n_db) return TQ_ERR_INVALID_ARG;
  if (nq > search_max_queries() || ctx->cfg.d != kD) return TQ_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15) || (reinterpret_cast<uintptr_t>(k_cache) & 15))
    return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}
}  // namespace

extern "C" tq_status tq_search_workspace_size(const tq_ctx* ctx, int nq, int n_db, int k_top, size_t* bytes) {
  if (!ctx || !bytes || nq < 1 || n_db < 1 || k_top < 0) return TQ_ERR_INVALID_ARG;
  *bytes = search_bytes(ctx, nq, n_db, k_top);
  return TQ_OK;
}

extern "C" tq_status tq_search(const tq_ctx* ctx, const void* q, tq_dtype dtype, int nq, const void* k_cache,
                               const int32_t* block_table, int num_pages, int n_db, int k_top,
                               float* top_scores, int32_t* top_index, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (!top_scores || !top_index) return TQ_ERR_INVALID_ARG;
  if (k_top < 1 || k_top > n_db || k_top > search_max_k()) return TQ_ERR_INVALID_ARG;
  tq_status st = search_check(ctx, q, dtype, nq, k_cache, block_table, num_pages, n_db, workspace);
  if (st != TQ_OK) return st;
  if (workspace_bytes < search_bytes(ctx, nq, n_db, k_top)) return TQ_ERR_WORKSPACE;
  DecodeArgs a = search_args(ctx, q, dtype, nq, workspace);
  char* extra = static_cast<char*>(workspace) + search_qrows_bytes(nq, ctx->cfg.m);
  const auto* kc = static_cast<const uint8_t*>(k_cache);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (search_tc_supported(ctx->kl, ctx->cfg.m, k_top))
    return cuda_status(launch_search_tc(a, kc, block_table, num_pages, n_db, k_top, top_scores, top_index, nullptr,
                                        extra, s));
  return cuda_status(launch_search(a, kc, block_table, num_pages, n_db, k_top, top_scores, top_index,
                                   reinterpret_cast<float*>(extra), s));
}

extern "C" tq_status tq_search_scores(const tq_ctx* ctx, const void* q, tq_dtype dtype, int nq, const void* k_cache,
                                      const int32_t* block_table, int num_pages, int n_db, int k_top, float* scores,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!scores || k_top < 1 || k_top > n_db || k_top > search_max_k()) return TQ_ERR_INVALID_ARG;
  tq_status st = search_check(ctx, q, dtype, nq, k_cache, block_table, num_pages, n_db, workspace);
  if (st != TQ_OK) return st;
  if (workspace_bytes < search_bytes(ctx, nq, n_db, 0)) return TQ_ERR_WORKSPACE;
  DecodeArgs a = search_args(ctx, q, dtype, nq, workspace);
  const auto* kc = static_cast<const uint8_t*>(k_cache);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (search_tc_supported(ctx->kl, ctx->cfg.m, k_top))
    return cuda_status(launch_search_tc(a, kc, block_table, num_pages, n_db, 1, nullptr, nullptr, scores, nullptr, s));
  return cuda_status(launch_search(a, kc, block_table, num_pages, n_db, 1, nullptr, nullptr, scores, s));
}
