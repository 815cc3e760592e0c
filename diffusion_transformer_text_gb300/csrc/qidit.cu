// C-ABI of the Qwen-Image-2.1 DiT step library: handle, weight store, pass
// orchestration and the host-contract entry points (declared in include/qidit.h).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <utility>
#include <string>
#include <vector>

#include "../../include/qidit.h"
#include "internal.h"

using qi::kBM;
using qi::kBN;
using qi::kFfn;
using qi::kHidden;
using qi::kMod;
using qi::kPatch;
using qi::kRopeCols;
using qi::kSspParts;
using qi::kTdim;
using qi::act_t;

namespace {

thread_local std::string g_last_error;

qi_status fail(qi_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define QI_CUDA(call)                                                                              \
  do {                                                                                             \
    cudaError_t e_ = (call);                                                                       \
    if (e_ != cudaSuccess)                                                                         \
      return fail(e_ == cudaErrorMemoryAllocation ? QI_ERR_OOM : QI_ERR_CUDA, "%s failed: %s (%s:%d)", \
                  #call, cudaGetErrorString(e_), __FILE__, __LINE__);                              \
  } while (0)

#define QI_TRY(expr)                  \
  do {                                \
    qi_status s_ = (expr);            \
    if (s_ != QI_OK) return s_;       \
  } while (0)

// ---------------------------------------------------------------- tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D 16-bit map over a row-major [rows, cols] matrix (fp16 unless `bf16`); box =
// box_rows x 64 columns (one 128-byte swizzle span), rows past `rows` read as zero.
qi_status make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   bool bf16 = false) {
  if (!encode_fn()) return fail(QI_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (cols * 2) % 16 != 0)
    return fail(QI_ERR_INVALID_ARG, "tensor map base or row pitch not 16-byte aligned");
  if (!qi::encode_map16(m, base, rows, cols, box_rows, bf16)) return fail(QI_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return QI_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Test hook (qi_debug_inject kind 1): when > 0, counts down device allocations
// and fails the one that brings it to zero.
std::atomic<int> g_fail_alloc{0};

cudaError_t dev_alloc(void** p, size_t bytes) {
  int n = g_fail_alloc.load();
  while (n > 0) {
    if (g_fail_alloc.compare_exchange_weak(n, n - 1)) {
      if (n == 1) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
      }
      break;
    }
  }
  return cudaMalloc(p, bytes);
}

// Lazy buffers: an allocation failure is QI_ERR_OOM, any other error QI_ERR_CUDA.
#define QI_ALLOC(ptr, bytes)                                                                          \
  do {                                                                                              \
    cudaError_t e_ = dev_alloc(reinterpret_cast<void**>(&(ptr)), (bytes));                            \
    if (e_ == cudaErrorMemoryAllocation) return fail(QI_ERR_OOM, "device allocation of %zu bytes failed", \
                                                     static_cast<size_t>(bytes));                        \
    if (e_ != cudaSuccess) return fail(QI_ERR_CUDA, "%s", cudaGetErrorString(e_));                     \
  } while (0)

}  // namespace

// ---------------------------------------------------------------- handle

struct qi_dit {
  int device = 0;
  int blocks = 0;
  int L_max = 0, N_max = 0, R_max = 0;
  int act_rows = 0;  // rows of the activation buffers: R_max, or 2 N_max for two-prompt guidance
  int num_sms = 0;
  bool loaded_global = false;
  std::vector<bool> loaded_block;

  // weights (one allocation)
  void* wmem = nullptr;
  uint16_t *t_w1, *t_b1, *t_w2, *t_b2, *mod_w, *mod_b, *txt_norm_w, *txt_w, *txt_b, *img_w, *img_b, *out_w, *out_b;
  struct Block {
    uint16_t* wqkv;  // [3*4096, 4096]: Q rows, K rows, V rows
    uint16_t* wo;    // [4096, 4096]
    uint16_t* wgu;   // [2*12288, 4096]: per 64-row group j, gate rows then up rows
    uint16_t* wd;    // [4096, 12288]
    CUtensorMap m_qkv, m_o, m_gu, m_d;
  };
  std::vector<Block> blk;
  CUtensorMap m_txt;

  // MXFP8 copies of the block weights (qi_dit_config.mxfp8): E4M3 bytes in the
  // layouts above plus their scale chunks, and the quantised A operand buffer
  bool has_mx = false;
  bool mx_on = false;  // the passes run the MXFP8 GEMMs (qi_dit_set_mxfp8)
  struct BlockMx {
    uint8_t *wqkv, *wo, *wgu, *wd;  // E4M3
    uint8_t *sqkv, *so, *sgu, *sd;  // scale chunks
    CUtensorMap m_qkv, m_o, m_gu, m_d;
  };
  std::vector<BlockMx> bmx;
  void* mxmem = nullptr;
  uint8_t* aq = nullptr;   // [act_rows, 12288] E4M3 activations (a GEMM's A operand)
  uint8_t* asf = nullptr;  // their scale chunks
  uint8_t* hq = nullptr;   // [act_rows, 12288] E4M3 SwiGLU output, written by the gate/up epilogue
  uint8_t* hsf = nullptr;

  // activations (one allocation)
  void* amem = nullptr;
  float* x = nullptr;      // [R_max, 4096] fp32 residual stream
  act_t* xa = nullptr;     // [R_max, 4096] fp16 modulated GEMM input
  float* ssp = nullptr;    // [R_max, 32] sum-of-squares partials (per 128 columns)
  float* out_wt = nullptr; // [4096, 64] the output head's weight, k-major fp32
  act_t* q = nullptr;      // [R_max, 4096]
  act_t* o = nullptr;      // [R_max, 4096] attention output
  act_t* h = nullptr;      // [R_max, 12288] SwiGLU hidden
  act_t* txt_a = nullptr;  // [L_max, 4096] text pre-norm output
  float* temb_e = nullptr; // [2, 256]
  float* temb_h = nullptr; // [2, 4096]
  float* temb = nullptr;   // [2, 4096]
  float* mod = nullptr;    // [2, 16384]: row 0 sampled t, row 1 t = 0
  int* err = nullptr;      // device error word
  act_t* kv = nullptr;     // [blocks][2][R_max][4096] fp16
  unsigned int* ovf = nullptr;  // weight values outside the fp16 range seen at load
  int slots = 1;           // text K/V slots: 1, or 2 for classifier-free guidance
  int cur_slot = 0;        // slot the running pass reads and writes
  int cache_L[2] = {-1, -1};  // per slot: L of the valid text K/V capture, -1 if none
  float* vel_pos = nullptr;   // [2 N_max, 64] guidance: conditional velocity rows, then (batch-2
                              // passes) the negative prompt's right after them
  float* vel_neg = nullptr;   // [N_max, 64] guidance: negative-prompt velocity (two-pass joint steps)

  // first-block cache, image rows only (allocated on first use)
  float* fbc_x0 = nullptr;            // [N_max, 4096] residual stream entering block 0
  float* fbc_x1 = nullptr;            // [N_max, 4096] leaving block 0
  float* fbc_r0[2] = {nullptr, nullptr};  // block 0's residual: reference and this pass
  float* fbc_rest = nullptr;          // [N_max, 4096] residual of blocks 1..last at the reference
  double2* fbc_part = nullptr;        // per-CTA sums of the change measure
  double* fbc_out = nullptr;          // {sum |r0 - ref|, sum |ref|}
  int fbc_ref = 0;                    // index of the reference in fbc_r0
  int fbc_N = -1;                     // N of the valid reference, -1 if none
  int fbc_L = -1;                     // L of the capture the reference was taken with

  // host-I/O staging (allocated on first use)
  float *st_img = nullptr, *st_txt = nullptr, *st_tc = nullptr, *st_ts = nullptr, *st_ic = nullptr,
        *st_is = nullptr, *st_vel = nullptr;

  int inject_stall = 0;  // test hook: the next block GEMM launch stalls its MMA issuer (bounded)

  int trace_block[2] = {-1, -1};
  float* trace_dst[2] = {nullptr, nullptr};
  float* range_out = nullptr;  // test hook: [blocks][QI_RANGE_KINDS] max |fp16 operand| (qi_dit_set_range_probe)

  unsigned prof_mask = 0;  // kernel classes timed with events (bit c = class c)
  int prof_stride = 1;     // block-level classes: only blocks b % prof_stride == 0
  struct ProfEv {
    int cls;
    cudaEvent_t a, b;
  };
  std::vector<ProfEv> prof_ev;
  size_t prof_used = 0;

  act_t* k_at(int slot, int b) { return kv + (static_cast<size_t>(slot) * blocks + b) * 2 * R_max * kHidden; }
  act_t* k_of(int b) { return k_at(cur_slot, b); }
  act_t* v_of(int b) { return k_of(b) + static_cast<size_t>(R_max) * kHidden; }
};

namespace {

enum PassMode { kJoint, kImage, kText };

struct ProfScope {
  qi_dit* d;
  cudaStream_t s;
  int cls;
  qi_dit::ProfEv* ev = nullptr;
  // block: the block index of a per-block launch group (-1 for the rest)
  ProfScope(qi_dit* d_, cudaStream_t s_, int c, int block = -1) : d(d_), s(s_), cls(c) {
    if (!((d->prof_mask >> c) & 1u)) return;
    if (block >= 0 && block % d->prof_stride != 0) return;
    if (d->prof_used == d->prof_ev.size()) {
      qi_dit::ProfEv e{c, nullptr, nullptr};
      cudaEventCreate(&e.a);
      cudaEventCreate(&e.b);
      d->prof_ev.push_back(e);
    }
    ev = &d->prof_ev[d->prof_used++];
    ev->cls = c;
    cudaEventRecord(ev->a, s);
  }
  ~ProfScope() {
    if (ev) cudaEventRecord(ev->b, s);
  }
};

qi_status check_device_word(qi_dit* d, cudaStream_t s) {
  int h = 0;
  QI_CUDA(cudaMemcpyAsync(&h, d->err, sizeof(int), cudaMemcpyDeviceToHost, s));
  QI_CUDA(cudaStreamSynchronize(s));
  if (h != 0) {
    QI_CUDA(cudaMemsetAsync(d->err, 0, sizeof(int), s));
    QI_CUDA(cudaStreamSynchronize(s));
    if (h == qi::kErrNonFinite) return fail(QI_ERR_NONFINITE, "the DiT pass produced a non-finite velocity");
    return fail(QI_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait expired (device code %d)", h);
  }
  return QI_OK;
}

// Operand-range test hook: fold max |a| over n fp16 values into the block's `kind` slot.
qi_status probe(qi_dit* d, int block, int kind, const act_t* a, long long n, cudaStream_t s) {
  if (!d->range_out || d->mx_on) return QI_OK;
  QI_CUDA(qi::launch_absmax_f16(a, n, d->range_out + block * QI_RANGE_KINDS + kind, s));
  return QI_OK;
}

qi_status compute_mod(qi_dit* d, float t, cudaStream_t s) {
  ProfScope ps(d, s, 5);
  QI_CUDA(qi::launch_timestep_embed(t, d->temb_e, s));
  QI_CUDA(qi::launch_gemv2(d->temb_e, kTdim, d->t_w1, d->t_b1, kHidden, d->temb_h, 0, d->err, true, s));
  QI_CUDA(qi::launch_gemv2(d->temb_h, kHidden, d->t_w2, d->t_b2, kHidden, d->temb, 1, d->err, true, s));
  QI_CUDA(qi::launch_gemv2(d->temb, kHidden, d->mod_w, d->mod_b, kMod, d->mod, 1, d->err, true, s));
  return QI_OK;
}

// One block over `R` activation rows. n_text = rows that are text (they come
// first); q_off = global index of activation row 0; Lk = keys image rows see.
// One GEMM of the block: fp16 operands, or (MXFP8 mode) the A operand `a16`
// quantised into the handle's E4M3 buffer first and the block's MXFP8 weights.
qi_status block_gemm(qi_dit* d, qi::EpiKind kind, const act_t* a16, int R, int K, const CUtensorMap& m_a16,
                     const CUtensorMap& m_w16, const CUtensorMap& m_w8, const uint8_t* w_sf, qi::GemmParams g,
                     cudaStream_t s, const uint8_t* a8 = nullptr, const uint8_t* a8_sf = nullptr) {
  if (!d->mx_on) {
    QI_CUDA(qi::launch_gemm(kind, m_a16, m_w16, g, d->num_sms, s));
    return QI_OK;
  }
  if (!a8) {
    // quantise the fp16 operand into the handle's buffer
    QI_CUDA(qi::launch_quant_mx(reinterpret_cast<const uint16_t*>(a16), false, R, K, d->aq, d->asf, s));
    a8 = d->aq;
    a8_sf = d->asf;
  }
  CUtensorMap m_a8;
  if (!qi::encode_map8(&m_a8, a8, R, K, 128)) return fail(QI_ERR_CUDA, "8-bit tensor map encoding failed");
  g.sfa = a8_sf;
  g.sfb = w_sf;
  QI_CUDA(qi::launch_gemm_mx(kind, m_a8, m_w8, g, d->num_sms, s));
  return QI_OK;
}

// The second prompt of a two-prompt (guidance) image-only pass: its image rows
// follow the first prompt's from row `split`; its text K/V sit in slot 1.
struct SecondPrompt {
  int split = 0;  // 0: a single-prompt pass
  int L = 0;
  const float* img_cos = nullptr;
  const float* img_sin = nullptr;
};

qi_status run_block(qi_dit* d, int b, int R, int n_text, int q_off, int L, int Lk, const float* txt_cos,
                    const float* txt_sin, const float* img_cos, const float* img_sin, cudaStream_t s,
                    const SecondPrompt& two = SecondPrompt{}) {
  qi_dit::Block& B = d->blk[b];
  qi_dit::BlockMx* BM = d->mx_on ? &d->bmx[b] : nullptr;
  CUtensorMap m_xa, m_o, m_h;
  QI_TRY(make_map(&m_xa, d->xa, R, kHidden, 128));
  QI_TRY(make_map(&m_o, d->o, R, kHidden, 128));
  QI_TRY(make_map(&m_h, d->h, R, kFfn, 128));

  qi::GemmParams p{};
  p.M = R;
  p.n_text = n_text;
  p.mod = d->mod;
  p.err = d->err;
  p.stall_test = d->inject_stall;  // one-shot: only this block's QKV GEMM carries it
  d->inject_stall = 0;
  // operand ranges (test hook) of single-prompt passes
  const bool rp = d->range_out && two.split == 0;
  const long long RH = static_cast<long long>(R) * kHidden;
  if (rp) QI_TRY(probe(d, b, 0, d->xa, RH, s));

  // QKV + 1/rms + RoPE -> Q and this block's K/V store
  {
    ProfScope ps(d, s, 0, b);
    qi::GemmParams g = p;
    g.N = 3 * kHidden;
    g.K = kHidden;
    g.ssp_in = d->ssp;
    g.q = d->q;
    g.k = d->k_of(b);
    g.v = d->v_of(b);
    g.kv_row_off = q_off;
    g.txt_cos = txt_cos;
    g.txt_sin = txt_sin;
    g.img_cos = img_cos;
    g.img_sin = img_sin;
    if (two.split > 0) {
      g.k = d->k_at(0, b);
      g.v = g.k + static_cast<size_t>(d->R_max) * kHidden;
      g.split_row = two.split;
      g.img_cos2 = two.img_cos;
      g.img_sin2 = two.img_sin;
      g.k2 = d->k_at(1, b);
      g.v2 = g.k2 + static_cast<size_t>(d->R_max) * kHidden;
      g.kv_row_off2 = two.L;
    }
    QI_TRY(block_gemm(d, qi::kEpiQkv, d->xa, R, kHidden, m_xa, B.m_qkv, BM ? BM->m_qkv : B.m_qkv,
                      BM ? BM->sqkv : nullptr, g, s));
    p.stall_test = 0;
  }
  if (rp) {
    QI_TRY(probe(d, b, 1, d->q, RH, s));
    QI_TRY(probe(d, b, 2, d->k_of(b) + static_cast<size_t>(q_off) * kHidden, RH, s));
    QI_TRY(probe(d, b, 3, d->v_of(b) + static_cast<size_t>(q_off) * kHidden, RH, s));
  }
  // block-causal attention
  {
    ProfScope ps(d, s, 1, b);
    qi::AttnParams a{};
    a.q = d->q;
    a.k = two.split > 0 ? d->k_at(0, b) : d->k_of(b);
    a.v = a.k + static_cast<size_t>(d->R_max) * kHidden;
    a.o = d->o;
    a.Rq = two.split > 0 ? two.split : R;
    a.q_off = q_off;
    a.L = L;
    a.Lk = Lk;
    a.err = d->err;
    if (d->mx_on) {
      // O straight into the out-projection's MXFP8 A operand (no fp16 copy)
      a.oq = d->aq;
      a.osf = d->asf;
      a.oq_row0 = 0;
      a.oq_groups = (R + kBM - 1) / kBM;
    }
    QI_CUDA(qi::launch_attention(a, s));
    if (two.split > 0) {
      // the second prompt's rows attend to its own text K/V (slot 1) and image K/V
      const size_t off = static_cast<size_t>(two.split) * kHidden;
      a.q = d->q + off;
      a.o = d->o + off;
      a.k = d->k_at(1, b);
      a.v = a.k + static_cast<size_t>(d->R_max) * kHidden;
      a.Rq = R - two.split;
      a.q_off = two.L;
      a.L = two.L;
      a.Lk = two.L + (R - two.split);
      a.oq_row0 = two.split;
      QI_CUDA(qi::launch_attention(a, s));
    }
  }
  if (rp) QI_TRY(probe(d, b, 4, d->o, RH, s));
  // out-projection: x += g1 * (o Wo^T); xa = fp16(x (1 + s2))
  {
    ProfScope ps(d, s, 2, b);
    qi::GemmParams g = p;
    g.N = kHidden;
    g.K = kHidden;
    g.x = d->x;
    g.xa = d->xa;
    g.ssp_out = d->ssp;
    g.resid_set = 0;
    g.gate_chunk = 1;
    g.scale_chunk = 2;
    QI_TRY(block_gemm(d, qi::kEpiResid, d->o, R, kHidden, m_o, B.m_o, BM ? BM->m_o : B.m_o, BM ? BM->so : nullptr, g,
                      s, BM ? d->aq : nullptr, BM ? d->asf : nullptr));
  }
  if (rp) QI_TRY(probe(d, b, 5, d->xa, RH, s));
  // gate/up + SwiGLU
  {
    ProfScope ps(d, s, 3, b);
    qi::GemmParams g = p;
    g.N = 2 * kFfn;
    g.K = kHidden;
    g.ssp_in = d->ssp;
    g.h = d->h;
    if (BM) {
      // h straight into the down GEMM's MXFP8 A operand
      g.hq = d->hq;
      g.hsf = d->hsf;
    }
    QI_TRY(block_gemm(d, qi::kEpiSwiglu, d->xa, R, kHidden, m_xa, B.m_gu, BM ? BM->m_gu : B.m_gu,
                      BM ? BM->sgu : nullptr, g, s));
  }
  if (rp) QI_TRY(probe(d, b, 6, d->h, static_cast<long long>(R) * kFfn, s));
  // down: x += g2 * (h Wd^T); xa = fp16(x (1 + s1)) for the next block
  {
    ProfScope ps(d, s, 4, b);
    qi::GemmParams g = p;
    g.N = kHidden;
    g.K = kFfn;
    g.x = d->x;
    g.xa = d->xa;
    g.ssp_out = d->ssp;
    g.resid_set = 0;
    g.gate_chunk = 3;
    g.scale_chunk = 0;
    QI_TRY(block_gemm(d, qi::kEpiResid, d->h, R, kFfn, m_h, B.m_d, BM ? BM->m_d : B.m_d, BM ? BM->sd : nullptr, g,
                      s, BM ? d->hq : nullptr, BM ? d->hsf : nullptr));
  }
  return QI_OK;
}

qi_status trace_copy(qi_dit* d, int at_block, int R, cudaStream_t s) {
  for (int i = 0; i < 2; ++i)
    if (d->trace_dst[i] && d->trace_block[i] == at_block)
      QI_CUDA(cudaMemcpyAsync(d->trace_dst[i], d->x, static_cast<size_t>(R) * kHidden * sizeof(float),
                              cudaMemcpyDeviceToDevice, s));
  return QI_OK;
}

// Rows of a pass. Joint: [text L | image N]; image: [image N] with the stored
// text K/V; text: [text L], no head.
struct PassRows {
  int n_text, n_img, R, q_off, Lk;
  PassRows(PassMode mode, int N, int L)
      : n_text(mode == kImage ? 0 : L),
        n_img(mode == kText ? 0 : N),
        R(n_text + n_img),
        q_off(mode == kImage ? L : 0),
        Lk(mode == kText ? L : L + N) {}
};

// Modulation rows and the input projections: x, xa, ssp for every row of the pass.
qi_status pass_embed(qi_dit* d, const PassRows& pr, const float* img, int N, const float* txt, int L, float t,
                     cudaStream_t s) {
  QI_TRY(compute_mod(d, t, s));
  {
    ProfScope ps(d, s, 5);
    if (pr.n_text > 0) {
      QI_CUDA(qi::launch_txt_prenorm(txt, L, d->txt_norm_w, d->txt_a, s));
      QI_TRY(probe(d, 0, 7, d->txt_a, static_cast<long long>(L) * kHidden, s));
    }
    if (pr.n_img > 0) {
      const size_t off = static_cast<size_t>(pr.n_text);
      QI_CUDA(qi::launch_img_in(img, N, d->img_w, d->img_b, d->mod, d->x + off * kHidden, d->xa + off * kHidden,
                                d->ssp + off * kSspParts, s));
    }
  }
  if (pr.n_text > 0) {
    ProfScope ps(d, s, 5);
    CUtensorMap m_a;
    QI_TRY(make_map(&m_a, d->txt_a, L, kHidden, 128));
    qi::GemmParams g{};
    g.M = L;
    g.N = kHidden;
    g.K = kHidden;
    g.n_text = L;
    g.mod = d->mod;
    g.err = d->err;
    g.x = d->x;
    g.xa = d->xa;
    g.ssp_out = d->ssp;
    g.bias = d->txt_b;
    g.resid_set = 1;
    g.gate_chunk = 1;
    g.scale_chunk = 0;
    QI_CUDA(qi::launch_gemm(qi::kEpiResid, m_a, d->m_txt, g, d->num_sms, s));
  }
  return QI_OK;
}

// Blocks b0 .. b1-1 over the pass's rows.
qi_status pass_blocks(qi_dit* d, const PassRows& pr, int b0, int b1, int L, const float* tc, const float* ts,
                      const float* ic, const float* is, cudaStream_t s) {
  for (int b = b0; b < b1; ++b) {
    QI_TRY(trace_copy(d, b, pr.R, s));
    QI_TRY(run_block(d, b, pr.R, pr.n_text, pr.q_off, L, pr.Lk, tc, ts, ic, is, s));
  }
  if (b1 == d->blocks) QI_TRY(trace_copy(d, d->blocks, pr.R, s));
  return QI_OK;
}

// Output head on the image rows (needs their ssp partials).
qi_status pass_head(qi_dit* d, const PassRows& pr, int N, float* vel, cudaStream_t s) {
  if (pr.n_img == 0) return QI_OK;
  ProfScope ps(d, s, 5);
  const size_t off = static_cast<size_t>(pr.n_text);
  QI_CUDA(qi::launch_head(d->x + off * kHidden, N, d->ssp + off * kSspParts, d->out_wt, d->out_b, vel, d->err, s));
  return QI_OK;
}

// Guidance, image rows only: both prompts' N image rows in one pass of 2N rows
// (first prompt, then second) over the text K/V in slots 0 and 1. Every GEMM
// row is computed as in a single-prompt pass, so each half equals that prompt's
// own image-only pass bit for bit. vel2: [2N, 64].
qi_status run_pass_two(qi_dit* d, const float* img, int N, float t, int L1, const float* ic1, const float* is1, int L2,
                       const float* ic2, const float* is2, float* vel2, cudaStream_t s) {
  d->cur_slot = 0;
  const int R = 2 * N;
  const size_t off = static_cast<size_t>(N);
  QI_TRY(compute_mod(d, t, s));
  {
    ProfScope ps(d, s, 5);
    QI_CUDA(qi::launch_img_in(img, N, d->img_w, d->img_b, d->mod, d->x, d->xa, d->ssp, s));
    QI_CUDA(qi::launch_img_in(img, N, d->img_w, d->img_b, d->mod, d->x + off * kHidden, d->xa + off * kHidden,
                              d->ssp + off * kSspParts, s));
  }
  SecondPrompt two;
  two.split = N;
  two.L = L2;
  two.img_cos = ic2;
  two.img_sin = is2;
  for (int b = 0; b < d->blocks; ++b) QI_TRY(run_block(d, b, R, 0, L1, L1, L1 + N, nullptr, nullptr, ic1, is1, s, two));
  {
    ProfScope ps(d, s, 5);
    QI_CUDA(qi::launch_head(d->x, R, d->ssp, d->out_wt, d->out_b, vel2, d->err, s));
  }
  return QI_OK;
}

qi_status run_pass(qi_dit* d, int slot, PassMode mode, const float* img, int N, const float* txt, int L, float t,
                   const float* tc, const float* ts, const float* ic, const float* is, float* vel,
                   cudaStream_t s) {
  d->cur_slot = slot;
  // a pass that rewrites slot 0's text K/V starts a new run for the first-block cache
  if (slot == 0 && mode != kImage) d->fbc_N = -1;
  const PassRows pr(mode, N, L);
  QI_TRY(pass_embed(d, pr, img, N, txt, L, t, s));
  QI_TRY(pass_blocks(d, pr, 0, d->blocks, L, tc, ts, ic, is, s));
  return pass_head(d, pr, N, vel, s);
}

// bf16 -> fp16 in place for tensor-core weights; synchronises `s`. A value beyond
// the fp16 range (|w| > 65504) makes the load fail.
qi_status convert_weights(qi_dit* d, std::initializer_list<std::pair<uint16_t*, size_t>> tensors, cudaStream_t s,
                          const char* who) {
  QI_CUDA(cudaMemsetAsync(d->ovf, 0, sizeof(unsigned int), s));
  for (auto& t : tensors) QI_CUDA(qi::launch_bf16_to_f16(t.first, t.second, d->ovf, s));
  unsigned int bad = 0;
  QI_CUDA(cudaMemcpyAsync(&bad, d->ovf, sizeof(bad), cudaMemcpyDeviceToHost, s));
  QI_CUDA(cudaStreamSynchronize(s));
  if (bad) return fail(QI_ERR_INVALID_ARG, "%s: %u weight values exceed the fp16 range (|w| > 65504)", who, bad);
  return QI_OK;
}

bool all_loaded(const qi_dit* d) {
  if (!d->loaded_global) return false;
  for (bool b : d->loaded_block)
    if (!b) return false;
  return true;
}

// Argument checks shared by the single-prompt step entry points. `vel` is the
// velocity output, or for the sampler step any non-NULL pointer.
qi_status step_checks(qi_dit* d, const char* who, const void* img, int N, const float* txt, int L, float t,
                      const float* tc, const float* ts, const float* ic, const float* is, const void* vel,
                      unsigned flags) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "%s: NULL handle", who);
  if (flags & ~(QI_STEP_USE_CACHE | QI_STEP_HOST_IO)) return fail(QI_ERR_INVALID_ARG, "%s: flags %u", who, flags);
  const bool use_cache = flags & QI_STEP_USE_CACHE;
  if (N < QI_N_MIN || N > d->N_max || L < QI_L_MIN || L > d->L_max)
    return fail(QI_ERR_SHAPE, "%s: N %d (max %d) L %d (max %d)", who, N, d->N_max, L, d->L_max);
  if (!img || !ic || !is || !vel) return fail(QI_ERR_INVALID_ARG, "%s: NULL image tensor", who);
  if (!use_cache && (!txt || !tc || !ts))
    return fail(QI_ERR_INVALID_ARG, "%s: joint pass needs txt_feats and txt_cos/txt_sin", who);
  if (use_cache && d->cache_L[0] != L)
    return fail(QI_ERR_STATE, "%s: USE_CACHE but the text K/V capture is for L=%d, not %d", who, d->cache_L[0], L);
  if (!all_loaded(d)) return fail(QI_ERR_STATE, "%s: weights not loaded", who);
  if (!std::isfinite(t)) return fail(QI_ERR_INVALID_ARG, "%s: timestep not finite", who);
  return QI_OK;
}

// Device staging for host-buffer steps (allocated on first use, held until destroy).
qi_status ensure_staging(qi_dit* d) {
  // each buffer once: a failed call leaves the ones it made for the next call
  if (!d->st_vel) QI_ALLOC(d->st_vel, (size_t)d->N_max * kPatch * 4);
  if (!d->st_ic) QI_ALLOC(d->st_ic, (size_t)d->N_max * kRopeCols * 4);
  if (!d->st_is) QI_ALLOC(d->st_is, (size_t)d->N_max * kRopeCols * 4);
  if (!d->st_txt) QI_ALLOC(d->st_txt, (size_t)d->L_max * kHidden * 4);
  if (!d->st_tc) QI_ALLOC(d->st_tc, (size_t)d->L_max * kRopeCols * 4);
  if (!d->st_ts) QI_ALLOC(d->st_ts, (size_t)d->L_max * kRopeCols * 4);
  if (!d->st_img) QI_ALLOC(d->st_img, (size_t)d->N_max * kPatch * 4);
  return QI_OK;
}

// Host -> staging copies of a step's inputs (the text ones only for a joint pass).
qi_status stage_inputs(qi_dit* d, const float* img, int N, const float* txt, int L, const float* tc, const float* ts,
                       const float* ic, const float* is, bool use_cache, cudaStream_t s) {
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
  QI_CUDA(cudaMemcpyAsync(d->st_img, img, (size_t)N * kPatch * 4, h2d, s));
  QI_CUDA(cudaMemcpyAsync(d->st_ic, ic, (size_t)N * kRopeCols * 4, h2d, s));
  QI_CUDA(cudaMemcpyAsync(d->st_is, is, (size_t)N * kRopeCols * 4, h2d, s));
  if (!use_cache) {
    QI_CUDA(cudaMemcpyAsync(d->st_txt, txt, (size_t)L * kHidden * 4, h2d, s));
    QI_CUDA(cudaMemcpyAsync(d->st_tc, tc, (size_t)L * kRopeCols * 4, h2d, s));
    QI_CUDA(cudaMemcpyAsync(d->st_ts, ts, (size_t)L * kRopeCols * 4, h2d, s));
  }
  return QI_OK;
}

}  // namespace

void qi::set_last_error(const char* msg) { g_last_error = msg; }

bool qi::encode_map16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || (cols * 2) % 16 != 0 || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool qi::encode_map8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || cols % 16 != 0 || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ================================================================ C ABI

extern "C" {

const char* qi_last_error(void) { return g_last_error.c_str(); }

size_t qi_kv_cache_bytes(int blocks, int L) {
  if (blocks <= 0 || L <= 0) return 0;
  return static_cast<size_t>(2) * blocks * L * kHidden * 2;
}

qi_status qi_dit_create(const qi_dit_config* cfg, int device, qi_dit** out) {
  if (!cfg || !out) return fail(QI_ERR_INVALID_ARG, "qi_dit_create: NULL argument");
  *out = nullptr;
  if (cfg->kv_slots < 0 || cfg->kv_slots > 2)
    return fail(QI_ERR_SHAPE, "qi_dit_create: kv_slots %d (0, 1 or 2)", cfg->kv_slots);
  if (cfg->blocks < 1 || cfg->blocks > QI_BLOCKS || cfg->L_max < QI_L_MIN || cfg->L_max > QI_L_MAX ||
      cfg->N_max < QI_N_MIN || cfg->N_max > QI_N_MAX)
    return fail(QI_ERR_SHAPE, "qi_dit_create: blocks %d L_max %d N_max %d out of range", cfg->blocks, cfg->L_max,
                cfg->N_max);
  QI_CUDA(cudaSetDevice(device));
  qi_dit* d = new qi_dit();
  d->device = device;
  d->blocks = cfg->blocks;
  d->L_max = cfg->L_max;
  d->N_max = cfg->N_max;
  d->R_max = cfg->L_max + cfg->N_max;
  d->act_rows = cfg->kv_slots == 2 ? std::max(d->R_max, 2 * cfg->N_max) : d->R_max;
  d->slots = cfg->kv_slots == 2 ? 2 : 1;
  d->loaded_block.assign(cfg->blocks, false);
  cudaDeviceGetAttribute(&d->num_sms, cudaDevAttrMultiProcessorCount, device);

  // ---- weights
  const size_t A = 256;
  struct Seg {
    uint16_t** p;
    size_t n;
  };
  std::vector<Seg> segs = {
      {&d->t_w1, (size_t)kHidden * kTdim}, {&d->t_b1, (size_t)kHidden},
      {&d->t_w2, (size_t)kHidden * kHidden}, {&d->t_b2, (size_t)kHidden},
      {&d->mod_w, (size_t)kMod * kHidden}, {&d->mod_b, (size_t)kMod},
      {&d->txt_norm_w, (size_t)kHidden}, {&d->txt_w, (size_t)kHidden * kHidden},
      {&d->txt_b, (size_t)kHidden}, {&d->img_w, (size_t)kHidden * kPatch},
      {&d->img_b, (size_t)kHidden}, {&d->out_w, (size_t)kPatch * kHidden},
      {&d->out_b, (size_t)kPatch},
  };
  d->blk.resize(cfg->blocks);
  for (auto& b : d->blk) {
    segs.push_back({&b.wqkv, (size_t)3 * kHidden * kHidden});
    segs.push_back({&b.wo, (size_t)kHidden * kHidden});
    segs.push_back({&b.wgu, (size_t)2 * kFfn * kHidden});
    segs.push_back({&b.wd, (size_t)kHidden * kFfn});
  }
  size_t wbytes = 0;
  for (auto& s : segs) wbytes += align_up(s.n * 2, A);
  cudaError_t e = dev_alloc(&d->wmem, wbytes);
  if (e != cudaSuccess) {
    delete d;
    return fail(QI_ERR_OOM, "qi_dit_create: weight store of %zu bytes: %s", wbytes, cudaGetErrorString(e));
  }
  {
    char* p = static_cast<char*>(d->wmem);
    for (auto& s : segs) {
      *s.p = reinterpret_cast<uint16_t*>(p);
      p += align_up(s.n * 2, A);
    }
  }

  // ---- activations and K/V store
  const size_t R = d->act_rows;
  struct ASeg {
    void** p;
    size_t bytes;
  };
  std::vector<ASeg> asegs = {
      {(void**)&d->x, R * kHidden * 4},   {(void**)&d->xa, R * kHidden * 2},
      {(void**)&d->ssp, R * kSspParts * 4}, {(void**)&d->q, R * kHidden * 2},
      {(void**)&d->o, R * kHidden * 2},   {(void**)&d->h, R * kFfn * 2},
      {(void**)&d->txt_a, (size_t)d->L_max * kHidden * 2}, {(void**)&d->temb_e, 2 * kTdim * 4},
      {(void**)&d->temb_h, 2 * kHidden * 4}, {(void**)&d->temb, 2 * kHidden * 4},
      {(void**)&d->mod, 2 * (size_t)kMod * 4}, {(void**)&d->err, 256}, {(void**)&d->ovf, 256},
      {(void**)&d->out_wt, (size_t)kHidden * kPatch * 4},
      {(void**)&d->kv, (size_t)d->slots * cfg->blocks * 2 * d->R_max * kHidden * 2},
      {(void**)&d->vel_pos, d->slots == 2 ? 2 * (size_t)d->N_max * kPatch * 4 : 0},
      {(void**)&d->vel_neg, d->slots == 2 ? (size_t)d->N_max * kPatch * 4 : 0},
  };
  size_t abytes = 0;
  for (auto& s : asegs) abytes += align_up(s.bytes, 1024);
  e = dev_alloc(&d->amem, abytes);
  if (e != cudaSuccess) {
    cudaFree(d->wmem);
    delete d;
    return fail(QI_ERR_OOM, "qi_dit_create: activations of %zu bytes: %s", abytes, cudaGetErrorString(e));
  }
  {
    char* p = static_cast<char*>(d->amem);
    for (auto& s : asegs) {
      *s.p = p;
      p += align_up(s.bytes, 1024);
    }
  }
  cudaMemset(d->amem, 0, abytes);

  // ---- MXFP8 weight copies and the quantised activation buffer
  if (cfg->mxfp8) {
    const size_t sq = (size_t)kHidden * kHidden;
    auto sf_bytes = [](size_t rows, size_t K) { return (rows + 127) / 128 * (K / 128) * 512; };
    const size_t per_block = align_up(3 * sq, 1024) + align_up(sq, 1024) + align_up(2 * (size_t)kFfn * kHidden, 1024) +
                             align_up((size_t)kHidden * kFfn, 1024) + align_up(sf_bytes(3 * kHidden, kHidden), 1024) +
                             align_up(sf_bytes(kHidden, kHidden), 1024) +
                             align_up(sf_bytes(2 * kFfn, kHidden), 1024) + align_up(sf_bytes(kHidden, kFfn), 1024);
    const size_t act = 2 * (align_up(R * kFfn, 1024) + align_up(sf_bytes(R, kFfn), 1024));
    e = dev_alloc(&d->mxmem, per_block * cfg->blocks + act);
    if (e != cudaSuccess) {
      cudaFree(d->amem);
      cudaFree(d->wmem);
      delete d;
      return fail(QI_ERR_OOM, "qi_dit_create: MXFP8 store: %s", cudaGetErrorString(e));
    }
    char* p = static_cast<char*>(d->mxmem);
    auto take = [&p](size_t n) {
      uint8_t* r = reinterpret_cast<uint8_t*>(p);
      p += align_up(n, 1024);
      return r;
    };
    d->bmx.resize(cfg->blocks);
    for (auto& b : d->bmx) {
      b.wqkv = take(3 * sq);
      b.wo = take(sq);
      b.wgu = take(2 * (size_t)kFfn * kHidden);
      b.wd = take((size_t)kHidden * kFfn);
      b.sqkv = take(sf_bytes(3 * kHidden, kHidden));
      b.so = take(sf_bytes(kHidden, kHidden));
      b.sgu = take(sf_bytes(2 * kFfn, kHidden));
      b.sd = take(sf_bytes(kHidden, kFfn));
    }
    d->aq = take(R * kFfn);
    d->asf = take(sf_bytes(R, kFfn));
    d->hq = take(R * kFfn);
    d->hsf = take(sf_bytes(R, kFfn));
    d->has_mx = true;
  }

  // ---- weight tensor maps (B operands: 128-row boxes for the CTA-pair fp16 GEMM,
  // 256-row boxes for the MXFP8 GEMM)
  const uint32_t bx = qi::kBoxRowsPair;
  qi_status st = make_map(&d->m_txt, d->txt_w, kHidden, kHidden, bx);
  for (int b = 0; st == QI_OK && b < cfg->blocks; ++b) {
    auto& B = d->blk[b];
    st = make_map(&B.m_qkv, B.wqkv, 3 * kHidden, kHidden, bx);
    if (st == QI_OK) st = make_map(&B.m_o, B.wo, kHidden, kHidden, bx);
    if (st == QI_OK) st = make_map(&B.m_gu, B.wgu, 2 * kFfn, kHidden, bx);
    if (st == QI_OK) st = make_map(&B.m_d, B.wd, kHidden, kFfn, bx);
    if (st == QI_OK && d->has_mx) {
      auto& M = d->bmx[b];
      if (!qi::encode_map8(&M.m_qkv, M.wqkv, 3 * kHidden, kHidden, 256) ||
          !qi::encode_map8(&M.m_o, M.wo, kHidden, kHidden, 256) ||
          !qi::encode_map8(&M.m_gu, M.wgu, 2 * kFfn, kHidden, 256) ||
          !qi::encode_map8(&M.m_d, M.wd, kHidden, kFfn, 256))
        st = fail(QI_ERR_CUDA, "qi_dit_create: 8-bit tensor map encoding failed");
    }
  }
  if (st != QI_OK) {
    if (d->mxmem) cudaFree(d->mxmem);
    cudaFree(d->amem);
    cudaFree(d->wmem);
    delete d;
    return st;
  }
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(d->amem);
    cudaFree(d->wmem);
    delete d;
    return fail(QI_ERR_CUDA, "qi_dit_create: %s", cudaGetErrorString(e));
  }
  *out = d;
  return QI_OK;
}

qi_status qi_dit_destroy(qi_dit* d) {
  if (!d) return QI_OK;
  cudaSetDevice(d->device);
  cudaDeviceSynchronize();
  for (auto& e : d->prof_ev) {
    cudaEventDestroy(e.a);
    cudaEventDestroy(e.b);
  }
  float* st[] = {d->st_img, d->st_txt, d->st_tc, d->st_ts, d->st_ic, d->st_is, d->st_vel,
                 d->fbc_x0, d->fbc_x1, d->fbc_r0[0], d->fbc_r0[1], d->fbc_rest};
  for (float* p : st)
    if (p) cudaFree(p);
  if (d->mxmem) cudaFree(d->mxmem);
  if (d->fbc_part) cudaFree(d->fbc_part);
  if (d->fbc_out) cudaFree(d->fbc_out);
  cudaFree(d->amem);
  cudaFree(d->wmem);
  delete d;
  return QI_OK;
}

qi_status qi_dit_load_global(qi_dit* d, const qi_global_weights* w, int src_on_device, qi_stream_t stream) {
  if (!d || !w) return fail(QI_ERR_INVALID_ARG, "qi_dit_load_global: NULL argument");
  const void* src[] = {w->t_w1, w->t_b1, w->t_w2, w->t_b2, w->mod_w, w->mod_b, w->txt_norm_w,
                       w->txt_w, w->txt_b, w->img_w, w->img_b, w->out_w, w->out_b};
  uint16_t* dst[] = {d->t_w1, d->t_b1, d->t_w2, d->t_b2, d->mod_w, d->mod_b, d->txt_norm_w,
                     d->txt_w, d->txt_b, d->img_w, d->img_b, d->out_w, d->out_b};
  const size_t n[] = {(size_t)kHidden * kTdim, kHidden, (size_t)kHidden * kHidden, kHidden,
                      (size_t)kMod * kHidden, kMod, kHidden, (size_t)kHidden * kHidden, kHidden,
                      (size_t)kHidden * kPatch, kHidden, (size_t)kPatch * kHidden, kPatch};
  for (int i = 0; i < 13; ++i)
    if (!src[i]) return fail(QI_ERR_INVALID_ARG, "qi_dit_load_global: tensor %d is NULL", i);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  const cudaMemcpyKind kind = src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
  for (int i = 0; i < 13; ++i) QI_CUDA(cudaMemcpyAsync(dst[i], src[i], n[i] * 2, kind, s));
  // the output head reads its weight as a k-major fp32 copy
  QI_CUDA(qi::launch_head_wt(d->out_w, d->out_wt, s));
  // the text projection runs on the tensor cores with fp16 operands
  QI_TRY(convert_weights(d, {{d->txt_w, (size_t)kHidden * kHidden}}, s, "qi_dit_load_global"));
  d->loaded_global = true;
  return QI_OK;
}

qi_status qi_dit_load_block(qi_dit* d, int block, const qi_block_weights* w, int src_on_device,
                            qi_stream_t stream) {
  if (!d || !w) return fail(QI_ERR_INVALID_ARG, "qi_dit_load_block: NULL argument");
  if (block < 0 || block >= d->blocks) return fail(QI_ERR_INVALID_ARG, "qi_dit_load_block: block %d", block);
  if (!w->wq || !w->wk || !w->wv || !w->wo || !w->wg || !w->wu || !w->wd)
    return fail(QI_ERR_INVALID_ARG, "qi_dit_load_block: a tensor is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  const cudaMemcpyKind kind = src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
  auto& B = d->blk[block];
  const size_t sq = (size_t)kHidden * kHidden;
  QI_CUDA(cudaMemcpyAsync(B.wqkv, w->wq, sq * 2, kind, s));
  QI_CUDA(cudaMemcpyAsync(B.wqkv + sq, w->wk, sq * 2, kind, s));
  QI_CUDA(cudaMemcpyAsync(B.wqkv + 2 * sq, w->wv, sq * 2, kind, s));
  QI_CUDA(cudaMemcpyAsync(B.wo, w->wo, sq * 2, kind, s));
  // gate/up interleave: 64-row groups, gate group j then up group j, so any 128
  // GEMM columns (a half tile) pair the gate and up rows of the same 64 hidden units
  constexpr int kGuRows = 64;
  const size_t grp = (size_t)kGuRows * kHidden * 2;  // bytes per 64-row group
  QI_CUDA(cudaMemcpy2DAsync(B.wgu, 2 * grp, w->wg, grp, grp, kFfn / kGuRows, kind, s));
  QI_CUDA(cudaMemcpy2DAsync(reinterpret_cast<char*>(B.wgu) + grp, 2 * grp, w->wu, grp, grp, kFfn / kGuRows, kind, s));
  QI_CUDA(cudaMemcpyAsync(B.wd, w->wd, (size_t)kHidden * kFfn * 2, kind, s));
  if (d->has_mx) {
    // from the bf16 values themselves, before they become fp16
    auto& M = d->bmx[block];
    QI_CUDA(qi::launch_quant_mx(B.wqkv, true, 3 * kHidden, kHidden, M.wqkv, M.sqkv, s));
    QI_CUDA(qi::launch_quant_mx(B.wo, true, kHidden, kHidden, M.wo, M.so, s));
    QI_CUDA(qi::launch_quant_mx(B.wgu, true, 2 * kFfn, kHidden, M.wgu, M.sgu, s));
    QI_CUDA(qi::launch_quant_mx(B.wd, true, kHidden, kFfn, M.wd, M.sd, s));
  }
  QI_TRY(convert_weights(d,
                         {{B.wqkv, 3 * sq}, {B.wo, sq}, {B.wgu, (size_t)2 * kFfn * kHidden}, {B.wd, (size_t)kHidden * kFfn}},
                         s, "qi_dit_load_block"));
  d->loaded_block[block] = true;
  return QI_OK;
}

qi_status qi_rope_axis_tables(float theta, float* cos0, float* sin0, float* cos1, float* sin1, float* cos2,
                              float* sin2, qi_stream_t stream) {
  if (!(theta > 1.f)) return fail(QI_ERR_INVALID_ARG, "qi_rope_axis_tables: theta %g", theta);
  QI_CUDA(qi::launch_rope_axis(theta, cos0, sin0, cos1, sin1, cos2, sin2, reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_rope_tables(int L, int h, int w, float theta, float* txt_cos, float* txt_sin, float* img_cos,
                         float* img_sin, qi_stream_t stream) {
  if (L < QI_L_MIN || L > QI_L_MAX || h < 1 || w < 1 || (long long)h * w > QI_N_MAX)
    return fail(QI_ERR_SHAPE, "qi_rope_tables: L %d h %d w %d out of range", L, h, w);
  // every position must fall inside the table range -1024..8191
  if (h - h / 2 > 1024 || w - w / 2 > 1024 || L > 8191)
    return fail(QI_ERR_SHAPE, "qi_rope_tables: positions leave the table range");
  if (!(theta > 1.f)) return fail(QI_ERR_INVALID_ARG, "qi_rope_tables: theta %g", theta);
  QI_CUDA(qi::launch_rope_tokens(L, h, w, theta, txt_cos, txt_sin, img_cos, img_sin,
                                 reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_flow_sigmas(int steps, int N, const qi_sched_params* p, float* sigmas, float* timesteps) {
  if (!sigmas || !timesteps) return fail(QI_ERR_INVALID_ARG, "qi_flow_sigmas: NULL output");
  // one step makes the terminal stretch 0/0 (its only sigma is 1), so at least two
  if (steps < 2 || N < 1) return fail(QI_ERR_SHAPE, "qi_flow_sigmas: steps %d (>= 2) N %d", steps, N);
  const qi_sched_params def = {0.5, 0.9, 256, 8192, 0.02, 1000};
  const qi_sched_params& c = p ? *p : def;
  if (c.max_seq == c.base_seq || c.shift_terminal >= 1.0)
    return fail(QI_ERR_INVALID_ARG, "qi_flow_sigmas: bad scheduler constants");
  // linspace(1, 1/steps, steps): start + i * step, last entry exactly the end point
  std::vector<double> s(steps);
  const double start = 1.0, stop = 1.0 / steps;
  if (steps == 1) {
    s[0] = start;
  } else {
    const double step = (stop - start) / (steps - 1);
    for (int i = 0; i < steps; ++i) s[i] = i * step + start;
    s[steps - 1] = stop;
  }
  const double m = (c.max_shift - c.base_shift) / (c.max_seq - c.base_seq);
  const double b = c.base_shift - m * c.base_seq;
  const double mu = N * m + b;
  const double e = std::exp(mu);
  for (int i = 0; i < steps; ++i) s[i] = e / (e + (1.0 / s[i] - 1.0));
  const double scale = (1.0 - s[steps - 1]) / (1.0 - c.shift_terminal);
  for (int i = 0; i < steps; ++i) s[i] = 1.0 - (1.0 - s[i]) / scale;
  for (int i = 0; i < steps; ++i) {
    timesteps[i] = static_cast<float>(s[i] * c.train_steps);
    sigmas[i] = static_cast<float>(s[i]);
  }
  sigmas[steps] = 0.f;
  return QI_OK;
}

qi_status qi_pack_noise(const float* z, int h, int w, float* x, qi_stream_t stream) {
  if (!z || !x) return fail(QI_ERR_INVALID_ARG, "qi_pack_noise: NULL argument");
  if (h < 1 || w < 1 || (long long)h * w > QI_N_MAX) return fail(QI_ERR_SHAPE, "qi_pack_noise: h %d w %d", h, w);
  QI_CUDA(qi::launch_pack_noise(z, h, w, x, reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_euler_update(float* x, const float* vel, int N, float sigma_i, float sigma_next, qi_stream_t stream) {
  if (!x || !vel) return fail(QI_ERR_INVALID_ARG, "qi_euler_update: NULL argument");
  if (N < 0) return fail(QI_ERR_SHAPE, "qi_euler_update: N %d", N);
  QI_CUDA(qi::launch_euler(x, vel, static_cast<long long>(N) * kPatch, sigma_i, sigma_next,
                           reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

// DPM++ 2M coefficients of step i, in float64 from the float32 sigmas, rounded once.
// lambda(sigma) = log(1 - sigma) - log(sigma) is only needed for the ratio of two
// step sizes; a and b need no logarithm (alpha = 1 - sigma).
qi_status qi_dpmpp2m_coeffs(const float* sigmas, int steps, int i, int* order, float* coeffs) {
  if (!sigmas || !order || !coeffs) return fail(QI_ERR_INVALID_ARG, "qi_dpmpp2m_coeffs: NULL argument");
  if (steps < 1) return fail(QI_ERR_SHAPE, "qi_dpmpp2m_coeffs: steps %d", steps);
  if (i < 0 || i >= steps) return fail(QI_ERR_INVALID_ARG, "qi_dpmpp2m_coeffs: step %d of %d", i, steps);
  const double s = sigmas[i], sn = sigmas[i + 1];
  const double sp = i > 0 ? static_cast<double>(sigmas[i - 1]) : 1.0;
  if (!(s <= 1.0 && sn >= 0.0 && sn < s && (i == 0 || (sp <= 1.0 && sp > s))))
    return fail(QI_ERR_INVALID_ARG, "qi_dpmpp2m_coeffs: sigmas around step %d are not decreasing within [0, 1]", i);
  if (sn == 0.0) {
    *order = 0;
    coeffs[0] = 0.f;
    coeffs[1] = 1.f;
    coeffs[2] = 1.f;
    coeffs[3] = 0.f;
    return QI_OK;
  }
  coeffs[0] = static_cast<float>(sn / s);
  coeffs[1] = static_cast<float>((s - sn) / s);
  if (i == 0 || sp >= 1.0) {
    *order = 1;
    coeffs[2] = 1.f;
    coeffs[3] = 0.f;
    return QI_OK;
  }
  auto lambda = [](double v) { return std::log1p(-v) - std::log(v); };
  const double h = lambda(sn) - lambda(s);
  const double h_prev = lambda(s) - lambda(sp);
  const double c1 = h / (2.0 * h_prev);
  *order = 2;
  coeffs[2] = static_cast<float>(1.0 + c1);
  coeffs[3] = static_cast<float>(c1);
  return QI_OK;
}

qi_status qi_dpmpp2m_update(float* x, const float* vel, float* d_prev, int N, const float* sigmas, int steps, int i,
                            qi_stream_t stream) {
  if (!x || !vel || !d_prev) return fail(QI_ERR_INVALID_ARG, "qi_dpmpp2m_update: NULL argument");
  if (N < 0) return fail(QI_ERR_SHAPE, "qi_dpmpp2m_update: N %d", N);
  int order = 0;
  float c[4];
  QI_TRY(qi_dpmpp2m_coeffs(sigmas, steps, i, &order, c));
  QI_CUDA(qi::launch_dpmpp2m(x, vel, d_prev, static_cast<long long>(N) * kPatch, sigmas[i], order, c[0], c[1], c[2],
                             c[3], reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_dit_step(qi_dit* d, const float* img_tokens, int N, const float* txt_feats, int L, float timestep,
                      const float* txt_cos, const float* txt_sin, const float* img_cos, const float* img_sin,
                      float* vel, unsigned flags, qi_stream_t stream) {
  QI_TRY(step_checks(d, "qi_dit_step", img_tokens, N, txt_feats, L, timestep, txt_cos, txt_sin, img_cos, img_sin, vel,
                     flags));
  const bool use_cache = flags & QI_STEP_USE_CACHE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));

  if (flags & QI_STEP_HOST_IO) {
    QI_TRY(ensure_staging(d));
    QI_TRY(stage_inputs(d, img_tokens, N, txt_feats, L, txt_cos, txt_sin, img_cos, img_sin, use_cache, s));
    QI_TRY(run_pass(d, 0, use_cache ? kImage : kJoint, d->st_img, N, d->st_txt, L, timestep, d->st_tc, d->st_ts,
                    d->st_ic, d->st_is, d->st_vel, s));
    QI_CUDA(cudaMemcpyAsync(vel, d->st_vel, (size_t)N * kPatch * 4, cudaMemcpyDeviceToHost, s));
    if (!use_cache) d->cache_L[0] = L;
    return check_device_word(d, s);
  }
  QI_TRY(run_pass(d, 0, use_cache ? kImage : kJoint, img_tokens, N, txt_feats, L, timestep, txt_cos, txt_sin,
                  img_cos, img_sin, vel, s));
  if (!use_cache) d->cache_L[0] = L;
  return QI_OK;
}

qi_status qi_dit_euler_step(qi_dit* d, float* x, int N, const float* txt_feats, int L, float timestep, float sigma_i,
                            float sigma_next, const float* txt_cos, const float* txt_sin, const float* img_cos,
                            const float* img_sin, float* vel_out, unsigned flags, qi_stream_t stream) {
  // vel_out may be NULL: the step then keeps the velocity in the handle's staging buffer
  QI_TRY(step_checks(d, "qi_dit_euler_step", x, N, txt_feats, L, timestep, txt_cos, txt_sin, img_cos, img_sin, x,
                     flags));
  if (!std::isfinite(sigma_i) || !std::isfinite(sigma_next))
    return fail(QI_ERR_INVALID_ARG, "qi_dit_euler_step: sigmas not finite");
  const bool use_cache = flags & QI_STEP_USE_CACHE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  const long long n = static_cast<long long>(N) * kPatch;

  if (flags & QI_STEP_HOST_IO) {
    QI_TRY(ensure_staging(d));
    QI_TRY(stage_inputs(d, x, N, txt_feats, L, txt_cos, txt_sin, img_cos, img_sin, use_cache, s));
    QI_TRY(run_pass(d, 0, use_cache ? kImage : kJoint, d->st_img, N, d->st_txt, L, timestep, d->st_tc, d->st_ts,
                    d->st_ic, d->st_is, d->st_vel, s));
    QI_CUDA(qi::launch_euler(d->st_img, d->st_vel, n, sigma_i, sigma_next, s));
    QI_CUDA(cudaMemcpyAsync(x, d->st_img, static_cast<size_t>(n) * 4, cudaMemcpyDeviceToHost, s));
    if (vel_out) QI_CUDA(cudaMemcpyAsync(vel_out, d->st_vel, static_cast<size_t>(n) * 4, cudaMemcpyDeviceToHost, s));
    if (!use_cache) d->cache_L[0] = L;
    return check_device_word(d, s);
  }
  float* vel = vel_out;
  if (!vel) {
    QI_TRY(ensure_staging(d));
    vel = d->st_vel;
  }
  QI_TRY(run_pass(d, 0, use_cache ? kImage : kJoint, x, N, txt_feats, L, timestep, txt_cos, txt_sin, img_cos, img_sin,
                  vel, s));
  QI_CUDA(qi::launch_euler(x, vel, n, sigma_i, sigma_next, s));
  if (!use_cache) d->cache_L[0] = L;
  return QI_OK;
}

qi_status qi_dit_step_cfg(qi_dit* d, const float* img_tokens, int N, float timestep, float guidance,
                          const float* pos_feats, int L_pos, const float* pos_txt_cos, const float* pos_txt_sin,
                          const float* pos_img_cos, const float* pos_img_sin, const float* neg_feats, int L_neg,
                          const float* neg_txt_cos, const float* neg_txt_sin, const float* neg_img_cos,
                          const float* neg_img_sin, float* vel, unsigned flags, qi_stream_t stream) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_step_cfg: NULL handle");
  if (flags & ~QI_STEP_USE_CACHE) return fail(QI_ERR_INVALID_ARG, "qi_dit_step_cfg: flags %u", flags);
  if (d->slots != 2) return fail(QI_ERR_STATE, "qi_dit_step_cfg: the handle was created with one K/V slot");
  const bool use_cache = flags & QI_STEP_USE_CACHE;
  if (N < QI_N_MIN || N > d->N_max || L_pos < QI_L_MIN || L_pos > d->L_max || L_neg < QI_L_MIN || L_neg > d->L_max)
    return fail(QI_ERR_SHAPE, "qi_dit_step_cfg: N %d L_pos %d L_neg %d (max %d, %d)", N, L_pos, L_neg, d->N_max,
                d->L_max);
  if (!img_tokens || !vel || !pos_img_cos || !pos_img_sin || !neg_img_cos || !neg_img_sin)
    return fail(QI_ERR_INVALID_ARG, "qi_dit_step_cfg: NULL image tensor");
  if (!use_cache && (!pos_feats || !pos_txt_cos || !pos_txt_sin || !neg_feats || !neg_txt_cos || !neg_txt_sin))
    return fail(QI_ERR_INVALID_ARG, "qi_dit_step_cfg: a joint pass needs both prompts and their tables");
  if (use_cache && (d->cache_L[0] != L_pos || d->cache_L[1] != L_neg))
    return fail(QI_ERR_STATE, "qi_dit_step_cfg: USE_CACHE but the captures are for L=%d/%d, not %d/%d", d->cache_L[0],
                d->cache_L[1], L_pos, L_neg);
  if (!all_loaded(d)) return fail(QI_ERR_STATE, "qi_dit_step_cfg: weights not loaded");
  if (!std::isfinite(timestep) || !std::isfinite(guidance))
    return fail(QI_ERR_INVALID_ARG, "qi_dit_step_cfg: timestep or guidance not finite");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  const float* vneg = d->vel_neg;
  if (use_cache) {
    // both prompts in one pass of 2N rows (batch 2)
    QI_TRY(run_pass_two(d, img_tokens, N, timestep, L_pos, pos_img_cos, pos_img_sin, L_neg, neg_img_cos, neg_img_sin,
                        d->vel_pos, s));
    vneg = d->vel_pos + static_cast<size_t>(N) * kPatch;
  } else {
    // joint passes capture each prompt's text K/V in its slot
    QI_TRY(run_pass(d, 0, kJoint, img_tokens, N, pos_feats, L_pos, timestep, pos_txt_cos, pos_txt_sin, pos_img_cos,
                    pos_img_sin, d->vel_pos, s));
    QI_TRY(run_pass(d, 1, kJoint, img_tokens, N, neg_feats, L_neg, timestep, neg_txt_cos, neg_txt_sin, neg_img_cos,
                    neg_img_sin, d->vel_neg, s));
  }
  d->cur_slot = 0;
  {
    ProfScope ps(d, s, 5);
    QI_CUDA(qi::launch_cfg_combine(d->vel_pos, vneg, guidance, vel, static_cast<long long>(N) * kPatch, s));
  }
  if (!use_cache) {
    d->cache_L[0] = L_pos;
    d->cache_L[1] = L_neg;
  }
  return QI_OK;
}

qi_status qi_dit_step_fbcache(qi_dit* d, const float* img_tokens, int N, const float* txt_feats, int L,
                              float timestep, const float* txt_cos, const float* txt_sin, const float* img_cos,
                              const float* img_sin, float threshold, float* vel, float* rel_change, int* skipped,
                              unsigned flags, qi_stream_t stream) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_step_fbcache: NULL handle");
  if (flags & ~QI_STEP_USE_CACHE) return fail(QI_ERR_INVALID_ARG, "qi_dit_step_fbcache: flags %u", flags);
  const bool use_cache = flags & QI_STEP_USE_CACHE;
  if (N < QI_N_MIN || N > d->N_max || L < QI_L_MIN || L > d->L_max)
    return fail(QI_ERR_SHAPE, "qi_dit_step_fbcache: N %d (max %d) L %d (max %d)", N, d->N_max, L, d->L_max);
  if (!img_tokens || !img_cos || !img_sin || !vel)
    return fail(QI_ERR_INVALID_ARG, "qi_dit_step_fbcache: NULL image tensor");
  if (!use_cache && (!txt_feats || !txt_cos || !txt_sin))
    return fail(QI_ERR_INVALID_ARG, "qi_dit_step_fbcache: joint pass needs txt_feats and txt_cos/txt_sin");
  if (use_cache && d->cache_L[0] != L)
    return fail(QI_ERR_STATE, "qi_dit_step_fbcache: USE_CACHE but the capture is for L=%d, not %d", d->cache_L[0], L);
  if (!all_loaded(d)) return fail(QI_ERR_STATE, "qi_dit_step_fbcache: weights not loaded");
  if (!std::isfinite(timestep) || std::isnan(threshold))
    return fail(QI_ERR_INVALID_ARG, "qi_dit_step_fbcache: timestep or threshold not a number");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  const size_t img_bytes = static_cast<size_t>(d->N_max) * kHidden * sizeof(float);
  const int grid = 4 * d->num_sms;
  if (!d->fbc_x0) {
    QI_ALLOC(d->fbc_x0, img_bytes);
    QI_ALLOC(d->fbc_x1, img_bytes);
    QI_ALLOC(d->fbc_r0[0], img_bytes);
    QI_ALLOC(d->fbc_r0[1], img_bytes);
    QI_ALLOC(d->fbc_rest, img_bytes);
    QI_ALLOC(d->fbc_part, static_cast<size_t>(grid) * sizeof(double2));
    QI_ALLOC(d->fbc_out, 2 * sizeof(double));
  }
  d->cur_slot = 0;
  const PassMode mode = use_cache ? kImage : kJoint;
  const PassRows pr(mode, N, L);
  const size_t off = static_cast<size_t>(pr.n_text) * kHidden;
  // a joint pass starts a new run: no reference; so does a different image size or prompt
  const bool have_ref = use_cache && d->fbc_N == N && d->fbc_L == L;

  QI_TRY(pass_embed(d, pr, img_tokens, N, txt_feats, L, timestep, s));
  QI_CUDA(cudaMemcpyAsync(d->fbc_x0, d->x + off, static_cast<size_t>(N) * kHidden * sizeof(float),
                          cudaMemcpyDeviceToDevice, s));
  QI_TRY(pass_blocks(d, pr, 0, 1, L, txt_cos, txt_sin, img_cos, img_sin, s));
  float* r0 = d->fbc_r0[d->fbc_ref ^ 1];
  {
    ProfScope ps(d, s, 5);
    QI_CUDA(qi::launch_fbc_residual(d->x + off, d->fbc_x0, have_ref ? d->fbc_r0[d->fbc_ref] : nullptr, r0,
                                    d->fbc_x1, N, grid, d->fbc_part, d->fbc_out, s));
  }
  double rel = INFINITY;
  if (have_ref) {
    double h[2] = {0.0, 0.0};
    QI_CUDA(cudaMemcpyAsync(h, d->fbc_out, sizeof(h), cudaMemcpyDeviceToHost, s));
    QI_CUDA(cudaStreamSynchronize(s));
    rel = h[1] > 0.0 ? h[0] / h[1] : (h[0] == 0.0 ? 0.0 : INFINITY);
  }
  const bool skip = have_ref && rel < static_cast<double>(threshold);
  if (skip) {
    ProfScope ps(d, s, 5);
    QI_CUDA(qi::launch_fbc_apply(d->x + off, d->fbc_rest, d->ssp + static_cast<size_t>(pr.n_text) * kSspParts, N, s));
  } else {
    QI_TRY(pass_blocks(d, pr, 1, d->blocks, L, txt_cos, txt_sin, img_cos, img_sin, s));
    ProfScope ps(d, s, 5);
    QI_CUDA(qi::launch_fbc_rest(d->x + off, d->fbc_x1, d->fbc_rest, N, grid, s));
    d->fbc_ref ^= 1;
    d->fbc_N = N;
    d->fbc_L = L;
  }
  QI_TRY(pass_head(d, pr, N, vel, s));
  if (!use_cache) d->cache_L[0] = L;
  if (rel_change) *rel_change = static_cast<float>(rel);
  if (skipped) *skipped = skip ? 1 : 0;
  return QI_OK;
}

qi_status qi_dit_fbcache_reset(qi_dit* d) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_fbcache_reset: NULL handle");
  d->fbc_N = -1;
  d->fbc_L = -1;
  return QI_OK;
}

qi_status qi_text_kv_capture(qi_dit* d, const float* txt_feats, int L, const float* txt_cos, const float* txt_sin,
                             qi_stream_t stream) {
  if (!d || !txt_feats || !txt_cos || !txt_sin) return fail(QI_ERR_INVALID_ARG, "qi_text_kv_capture: NULL argument");
  if (L < QI_L_MIN || L > d->L_max) return fail(QI_ERR_SHAPE, "qi_text_kv_capture: L %d (max %d)", L, d->L_max);
  if (!all_loaded(d)) return fail(QI_ERR_STATE, "qi_text_kv_capture: weights not loaded");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  QI_TRY(run_pass(d, 0, kText, nullptr, 0, txt_feats, L, 0.f, txt_cos, txt_sin, nullptr, nullptr, nullptr, s));
  d->cache_L[0] = L;
  return QI_OK;
}

qi_status qi_dit_check(qi_dit* d, qi_stream_t stream) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_check: NULL handle");
  QI_CUDA(cudaSetDevice(d->device));
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(QI_ERR_CUDA, "qi_dit_check: %s", cudaGetErrorString(e));
  return check_device_word(d, reinterpret_cast<cudaStream_t>(stream));
}

qi_status qi_dit_block_forward(qi_dit* d, int block, float* hidden, int L, int N, float t_img, const float* cos,
                               const float* sin, qi_stream_t stream) {
  if (!d || !hidden || !cos || !sin) return fail(QI_ERR_INVALID_ARG, "qi_dit_block_forward: NULL argument");
  if (block < 0 || block >= d->blocks) return fail(QI_ERR_INVALID_ARG, "qi_dit_block_forward: block %d", block);
  if (L < 0 || N < 0 || L + N < 1 || L > d->L_max || N > d->N_max)
    return fail(QI_ERR_SHAPE, "qi_dit_block_forward: L %d N %d", L, N);
  if (!d->loaded_global || !d->loaded_block[block]) return fail(QI_ERR_STATE, "qi_dit_block_forward: not loaded");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  const int R = L + N;
  d->cur_slot = 0;
  QI_CUDA(cudaMemcpyAsync(d->x, hidden, (size_t)R * kHidden * 4, cudaMemcpyDeviceToDevice, s));
  QI_TRY(compute_mod(d, t_img, s));
  QI_CUDA(qi::launch_block_prep(d->x, R, L, d->mod, d->xa, d->ssp, s));
  QI_TRY(run_block(d, block, R, L, 0, L, R, cos, sin, cos + (size_t)L * kRopeCols, sin + (size_t)L * kRopeCols, s));
  QI_CUDA(cudaMemcpyAsync(hidden, d->x, (size_t)R * kHidden * 4, cudaMemcpyDeviceToDevice, s));
  return QI_OK;
}

qi_status qi_dit_read_kv(qi_dit* d, int block, int row0, int rows, uint16_t* k_out, uint16_t* v_out,
                         qi_stream_t stream) {
  if (!d || !k_out || !v_out) return fail(QI_ERR_INVALID_ARG, "qi_dit_read_kv: NULL argument");
  if (block < 0 || block >= d->blocks) return fail(QI_ERR_INVALID_ARG, "qi_dit_read_kv: block %d", block);
  if (row0 < 0 || rows < 0 || row0 + rows > d->R_max)
    return fail(QI_ERR_SHAPE, "qi_dit_read_kv: rows [%d, %d) past %d", row0, row0 + rows, d->R_max);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  QI_CUDA(cudaSetDevice(d->device));
  const size_t bytes = (size_t)rows * kHidden * 2;
  d->cur_slot = 0;
  QI_CUDA(cudaMemcpyAsync(k_out, d->k_of(block) + (size_t)row0 * kHidden, bytes, cudaMemcpyDeviceToDevice, s));
  QI_CUDA(cudaMemcpyAsync(v_out, d->v_of(block) + (size_t)row0 * kHidden, bytes, cudaMemcpyDeviceToDevice, s));
  return QI_OK;
}

qi_status qi_gemm_bf16(qi_dit* d, const uint16_t* A, const uint16_t* B, float* D, int M, int N, int K,
                       qi_stream_t stream) {
  if (!d || !A || !B || !D) return fail(QI_ERR_INVALID_ARG, "qi_gemm_bf16: NULL argument");
  if (M < 1 || N < kBN || N % kBN != 0 || K < qi::kBK || K % qi::kBK != 0)
    return fail(QI_ERR_SHAPE, "qi_gemm_bf16: M %d N %d K %d", M, N, K);
  CUtensorMap ma, mb;
  QI_TRY(make_map(&ma, A, M, K, 128, true));
  QI_TRY(make_map(&mb, B, N, K, qi::kBoxRowsPair, true));
  qi::GemmParams g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.d = D;
  g.err = d->err;
  QI_CUDA(cudaSetDevice(d->device));
  QI_CUDA(qi::launch_gemm(qi::kEpiF32, ma, mb, g, d->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_debug_inject(qi_dit* d, int kind, int arg) {
  switch (kind) {
    case 0:
      g_fail_alloc.store(0);
      if (d) d->inject_stall = 0;
      return QI_OK;
    case 1:
      if (arg < 1) return fail(QI_ERR_INVALID_ARG, "qi_debug_inject: allocation index %d (>= 1)", arg);
      g_fail_alloc.store(arg);
      return QI_OK;
    case 2:
      if (!d) return fail(QI_ERR_INVALID_ARG, "qi_debug_inject: kind 2 needs a handle");
      d->inject_stall = 1;
      return QI_OK;
  }
  return fail(QI_ERR_INVALID_ARG, "qi_debug_inject: kind %d", kind);
}

qi_status qi_dit_set_mxfp8(qi_dit* d, int on) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_set_mxfp8: NULL handle");
  if (on && !d->has_mx) return fail(QI_ERR_STATE, "qi_dit_set_mxfp8: the handle was created without mxfp8");
  if (d->mx_on != (on != 0)) {
    // text K/V and the first-block cache's reference were made by the other arithmetic
    d->cache_L[0] = d->cache_L[1] = -1;
    d->fbc_N = -1;
  }
  d->mx_on = on != 0;
  return QI_OK;
}

qi_status qi_quant_mxfp8(const uint16_t* in, int in_is_bf16, int rows, int K, uint8_t* q, uint8_t* sf,
                         qi_stream_t stream) {
  if (!in || !q || !sf) return fail(QI_ERR_INVALID_ARG, "qi_quant_mxfp8: NULL argument");
  if (rows < 1 || K < 128 || K % 128 != 0) return fail(QI_ERR_SHAPE, "qi_quant_mxfp8: rows %d K %d", rows, K);
  if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(q) & 15))
    return fail(QI_ERR_INVALID_ARG, "qi_quant_mxfp8: in and q must be 16-byte aligned");
  QI_CUDA(qi::launch_quant_mx(in, in_is_bf16 != 0, rows, K, q, sf, reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_gemm_mxfp8(qi_dit* d, const uint8_t* A, const uint8_t* A_sf, const uint8_t* B, const uint8_t* B_sf,
                        float* D, int M, int N, int K, qi_stream_t stream) {
  if (!d || !A || !A_sf || !B || !B_sf || !D) return fail(QI_ERR_INVALID_ARG, "qi_gemm_mxfp8: NULL argument");
  if (M < 1 || N < kBN || N % kBN != 0 || K < 128 || K % 128 != 0)
    return fail(QI_ERR_SHAPE, "qi_gemm_mxfp8: M %d N %d K %d", M, N, K);
  if ((reinterpret_cast<uintptr_t>(A_sf) & 15) || (reinterpret_cast<uintptr_t>(B_sf) & 15) ||
      (reinterpret_cast<uintptr_t>(D) & 15))
    return fail(QI_ERR_INVALID_ARG, "qi_gemm_mxfp8: scale chunks and D must be 16-byte aligned");
  CUtensorMap ma, mb;
  if (!qi::encode_map8(&ma, A, M, K, 128) || !qi::encode_map8(&mb, B, N, K, 256))
    return fail(QI_ERR_INVALID_ARG, "qi_gemm_mxfp8: tensor map encoding failed (alignment?)");
  qi::GemmParams g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.d = D;
  g.err = d->err;
  g.sfa = A_sf;
  g.sfb = B_sf;
  QI_CUDA(cudaSetDevice(d->device));
  QI_CUDA(qi::launch_gemm_mx(qi::kEpiF32, ma, mb, g, d->num_sms, reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_attention_f16(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, int Rq, int q_off,
                            int L, int Lk, qi_stream_t stream) {
  if (!q || !k || !v || !o) return fail(QI_ERR_INVALID_ARG, "qi_attention_f16: NULL argument");
  if (Rq < 0 || q_off < 0 || L < 0 || Lk < 1 || L > Lk || q_off + Rq > Lk)
    return fail(QI_ERR_SHAPE, "qi_attention_f16: Rq %d q_off %d L %d Lk %d", Rq, q_off, L, Lk);
  qi::AttnParams a{};
  a.q = reinterpret_cast<const act_t*>(q);
  a.k = reinterpret_cast<const act_t*>(k);
  a.v = reinterpret_cast<const act_t*>(v);
  a.o = reinterpret_cast<act_t*>(o);
  a.Rq = Rq;
  a.q_off = q_off;
  a.L = L;
  a.Lk = Lk;
  QI_CUDA(qi::launch_attention(a, reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_gemv_bf16(const float* x, int in_dim, const uint16_t* W, const uint16_t* b, int out_dim, float* y,
                       int silu_in, qi_stream_t stream) {
  if (!x || !W || !b || !y) return fail(QI_ERR_INVALID_ARG, "qi_gemv_bf16: NULL argument");
  if (out_dim < 1 || (in_dim != kTdim && in_dim != kHidden))
    return fail(QI_ERR_SHAPE, "qi_gemv_bf16: in_dim %d (256 or 4096) out_dim %d", in_dim, out_dim);
  QI_CUDA(qi::launch_gemv2(x, in_dim, W, b, out_dim, y, silu_in ? 1 : 0, nullptr, false,
                           reinterpret_cast<cudaStream_t>(stream)));
  return QI_OK;
}

qi_status qi_dit_set_trace(qi_dit* d, int slot, int block, float* dst) {
  if (!d || slot < 0 || slot > 1) return fail(QI_ERR_INVALID_ARG, "qi_dit_set_trace: bad handle or slot");
  if (dst && (block < 0 || block > d->blocks)) return fail(QI_ERR_INVALID_ARG, "qi_dit_set_trace: block %d", block);
  d->trace_block[slot] = dst ? block : -1;
  d->trace_dst[slot] = dst;
  return QI_OK;
}

qi_status qi_dit_set_range_probe(qi_dit* d, float* out) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_set_range_probe: NULL handle");
  if (out && (reinterpret_cast<uintptr_t>(out) & 3)) return fail(QI_ERR_INVALID_ARG, "qi_dit_set_range_probe: alignment");
  d->range_out = out;
  return QI_OK;
}

qi_status qi_dit_profile(qi_dit* d, int enable) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_profile: NULL handle");
  d->prof_mask = enable != 0 ? (1u << QI_PROF_CLASSES) - 1u : 0u;
  d->prof_stride = 1;
  d->prof_used = 0;
  return QI_OK;
}

qi_status qi_dit_profile_classes(qi_dit* d, unsigned mask, int block_stride) {
  if (!d) return fail(QI_ERR_INVALID_ARG, "qi_dit_profile_classes: NULL handle");
  if (mask >> QI_PROF_CLASSES) return fail(QI_ERR_INVALID_ARG, "qi_dit_profile_classes: mask 0x%x has bits past class %d",
                                            mask, QI_PROF_CLASSES - 1);
  if (block_stride < 1) return fail(QI_ERR_INVALID_ARG, "qi_dit_profile_classes: block_stride %d < 1", block_stride);
  d->prof_mask = mask;
  d->prof_stride = block_stride;
  d->prof_used = 0;
  return QI_OK;
}

qi_status qi_dit_profile_read(qi_dit* d, double* ms, long long* launches) {
  if (!d || !ms || !launches) return fail(QI_ERR_INVALID_ARG, "qi_dit_profile_read: NULL argument");
  for (int c = 0; c < QI_PROF_CLASSES; ++c) {
    ms[c] = 0.0;
    launches[c] = 0;
  }
  QI_CUDA(cudaSetDevice(d->device));
  for (size_t i = 0; i < d->prof_used; ++i) {
    auto& e = d->prof_ev[i];
    QI_CUDA(cudaEventSynchronize(e.b));
    float t = 0.f;
    QI_CUDA(cudaEventElapsedTime(&t, e.a, e.b));
    ms[e.cls] += t;
    launches[e.cls] += 1;
  }
  d->prof_used = 0;
  return QI_OK;
}

}  // extern "C"
