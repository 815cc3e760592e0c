// Declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

namespace qi {

constexpr int kHidden = 4096;
constexpr int kHeads = 32;
constexpr int kHeadDim = 128;
constexpr int kFfn = 12288;
constexpr int kMod = 4 * kHidden;
constexpr int kPatch = 64;
constexpr int kTdim = 256;
constexpr int kRopeCols = 64;
constexpr float kEps = 1e-6f;

// Codes a kernel writes into the device error word (first error wins).
enum DeviceError : int {
  kErrNone = 0,
  kErrTimeoutProducer = 1,  // a bounded mbarrier wait expired in a TMA producer
  kErrTimeoutMma = 2,       // ... in an MMA issuer
  kErrTimeoutEpilogue = 3,  // ... in an epilogue / softmax warp
  kErrTimeoutDrain = 4,     // ... while draining copies or MMAs before exit
  kErrNonFinite = 5,        // the output head produced a non-finite velocity
};

// Tensor-core operands of the DiT pass (GEMM A and B, Q/K/V, P, O) are fp16:
// the bf16 weights convert to fp16 exactly (except values below 2^-14, which
// lose < 2^-25), and fp16's 11-bit significand keeps the rounding of the
// activations 8x smaller than bf16's at the same tensor-core rate.
// Accumulation is fp32 throughout; the residual stream is fp32.
using act_t = __half;

// GEMM tile: 128 rows x 256 columns per CTA, K in steps of 64 (one 128-byte
// swizzle span of 16-bit elements). Sum-of-squares partials are kept per
// 128 columns, so that a tile split into two 128-column halves (the last
// wave of some GEMMs) writes its own partials; consumers add them in index order.
// The fp16 / bf16 GEMMs run on CTA pairs (256 x 256 per pair, 128 rows per CTA);
// each CTA loads half of the 256 B rows, so their B tensor maps use 128-row
// boxes (kBoxRowsPair). The MXFP8 GEMM runs one CTA per tile (256-row B boxes).
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kBoxRowsPair = kBN / 2;
constexpr int kSspCols = 128;                   // columns per sum-of-squares partial
constexpr int kSspParts = kHidden / kSspCols;  // 32 partial sums per row

enum EpiKind : int {
  kEpiQkv = 0,     // row scale 1/rms, RoPE on Q and K, fp16 Q / K / V stores
  kEpiResid = 1,   // residual update (+ gate) or bias set, fp16 modulated copy, sum of squares
  kEpiSwiglu = 2,  // row scale 1/rms, silu(gate) * up, fp16 store
  kEpiF32 = 3,     // plain fp32 store of D (test hooks, bf16 operands)
};

struct GemmParams {
  int M, N, K;
  int n_text;          // activation rows < n_text are text rows (t = 0 modulation row)
  const float* mod;    // [2][kMod]: row 0 for the sampled t, row 1 for t = 0
  const float* ssp_in; // [M][kSspParts] sum-of-squares partials of the GEMM's A rows
  // kEpiQkv
  act_t* q;
  act_t* k;
  act_t* v;
  int kv_row_off;      // K/V store row = activation row + kv_row_off
  const float* txt_cos;
  const float* txt_sin;
  const float* img_cos;
  const float* img_sin;
  // two prompts in one pass (guidance): if split_row > 0, rows >= split_row are the
  // second prompt's image rows: RoPE rows from img_cos2 / img_sin2 and K/V into
  // k2 / v2 at row (row - split_row) + kv_row_off2
  int split_row;
  const float* img_cos2;
  const float* img_sin2;
  act_t* k2;
  act_t* v2;
  int kv_row_off2;
  // kEpiSwiglu
  act_t* h;
  uint8_t* hq;   // MXFP8 (if set): h written as E4M3 codes [M][kFfn] and scales (hsf) instead of fp16
  uint8_t* hsf;
  // kEpiResid
  float* x;                 // fp32 residual stream [M][kHidden]
  act_t* xa;                // fp16(x * (1 + scale)) for the next GEMM
  float* ssp_out;           // [M][kSspParts]
  const uint16_t* bias;     // set mode: x = acc + bias (bf16 bits)
  int resid_set;            // 1: x = acc + bias; 0: x += gate * acc
  int gate_chunk;           // modulation chunk used as gate (0..3)
  int scale_chunk;          // modulation chunk used as (1 + scale) for xa
  float* d;                 // kEpiF32: D [M][N]
  int* err;                 // device error word
  // MXFP8 variant: scale chunks of A (ceil(M/128) row groups) and B (N/128 groups)
  const uint8_t* sfa;
  const uint8_t* sfb;
  // set by the launcher: tiles from this index on run as two 128-column halves
  int tail_start;
  // test hook: the MMA issuer first waits on a barrier nothing arrives on, so its
  // bounded wait expires (the launch reports kErrTimeoutMma and winds down)
  int stall_test;
};

// Launch one persistent tcgen05 GEMM D[M,N] = A[M,K] * B[N,K]^T with the
// epilogue `kind`. A and B maps are 2-D 16-bit maps with box {64, 128} /
// {64, 256}; the operands are fp16 for the DiT epilogues and bf16 for kEpiF32.
// Launch with programmatic stream serialization: the kernel's set-up (barrier
// initialisation, TMEM allocation, tensor-map prefetch) overlaps the end of the
// previous kernel in the stream. Only kernels that execute grid_dep_wait()
// before touching any activation (read or write) are launched this way, so each
// one still sees all earlier work complete; other kernels launch normally.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) holds for the current device
// only, so a launcher remembers per device ordinal (bit d of `done`; devices 64
// and up set it on every launch) whether it already raised the kernel's limit.
template <typename... KArgs>
cudaError_t ensure_smem_limit(void (*kernel)(KArgs...), int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

cudaError_t launch_gemm(EpiKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                        int grid_ctas, cudaStream_t stream);

// The MXFP8 variant: A and B maps are 2-D 8-bit maps with box {128, 128} /
// {128, 256}; p.sfa / p.sfb hold the UE8M0 scale chunks (layout in gemm.cu,
// written by launch_quant_mx). K must be a multiple of 128.
cudaError_t launch_gemm_mx(EpiKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                           int grid_ctas, cudaStream_t stream);

// 2-D 8-bit map over a row-major [rows, cols] byte matrix, box = box_rows x 128
// columns with 128-byte swizzle (qidit.cu).
bool encode_map8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// MXFP8 quantisation of a row-major [rows, K] 16-bit matrix (bf16 bits if `bf16`,
// else fp16) along K: q [rows, K] E4M3 bytes and the scale chunks for
// ceil(rows / 128) row groups (kernels_small.cu).
cudaError_t launch_quant_mx(const uint16_t* in, bool bf16, int rows, int K, uint8_t* q, uint8_t* sf,
                            cudaStream_t s);

struct AttnParams {
  const act_t* q;  // [Rq][kHidden], query row r has global index r + q_off
  const act_t* k;  // [Lk][kHidden], key rows 0..Lk-1 (text first)
  const act_t* v;
  act_t* o;        // [Rq][kHidden]
  int Rq;
  int q_off;
  int L;           // text rows: global index < L
  int Lk;          // keys visible to image rows
  int* err;        // device error word (may be null)
  // MXFP8 (if oq is set): O written as E4M3 codes and scales for the out-projection
  // instead of fp16 o; query row r is row oq_row0 + r of that A operand
  uint8_t* oq;
  uint8_t* osf;
  int oq_row0;
  int oq_groups;   // ceil(A operand rows / 128)
};

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream);

// 2-D 16-bit TMA map over a row-major [rows, cols] matrix, box = box_rows x 64
// columns with 128-byte swizzle; rows past `rows` read as zero (qidit.cu).
bool encode_map16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, bool bf16);

// Small kernels (kernels_small.cu)
cudaError_t launch_timestep_embed(float t, float* e, cudaStream_t s);
// y[r][o] = W[o] . act(x[r]) + b[o], r = 0, 1 (x [2][in_dim] fp32, W [out_dim][in_dim]
// bf16, act = silu if silu_in); in_dim = 4096 takes the streamed kernel (W and x
// 16-byte aligned), which reports a bounded wait's expiry in `err` (may be null).
// weights_preloaded: W was complete before the previous kernel in the stream began
// (the handle's weight store, written by copies at load), so the streamed kernel
// is launched dependent on that kernel and starts reading W while it finishes.
cudaError_t launch_gemv2(const float* x, int in_dim, const uint16_t* W, const uint16_t* b, int out_dim, float* y,
                         int silu_in, int* err, bool weights_preloaded, cudaStream_t s);
cudaError_t launch_txt_prenorm(const float* txt, int L, const uint16_t* w, act_t* out, cudaStream_t s);
cudaError_t launch_img_in(const float* img, int N, const uint16_t* W, const uint16_t* b, const float* mod,
                          float* x, act_t* xa, float* ssp, cudaStream_t s);
// wt: the head weight as a k-major fp32 copy [4096][64] (launch_head_wt, once at load)
cudaError_t launch_head(const float* x, int N, const float* ssp, const float* wt, const uint16_t* b, float* vel,
                        int* err, cudaStream_t s);
cudaError_t launch_head_wt(const uint16_t* W, float* wt, cudaStream_t s);
cudaError_t launch_block_prep(const float* x, int R, int n_text, const float* mod, act_t* xa, float* ssp,
                              cudaStream_t s);
cudaError_t launch_euler(float* x, const float* vel, long long n, float s_i, float s_next, cudaStream_t s);
cudaError_t launch_dpmpp2m(float* x, const float* vel, float* dprev, long long n, float sigma_i, int order, float a,
                           float b, float c0, float c1, cudaStream_t s);
cudaError_t launch_rope_axis(float theta, float* c0, float* s0, float* c1, float* s1, float* c2, float* s2,
                             cudaStream_t s);
cudaError_t launch_rope_tokens(int L, int h, int w, float theta, float* tc, float* ts, float* ic, float* is,
                               cudaStream_t s);
cudaError_t launch_pack_noise(const float* z, int h, int w, float* x, cudaStream_t s);
// First-block cache. residual: r0 = x1 - x0 and x1c = x1 over rows x 4096; when ref is
// not null also out = {sum |r0 - ref|, sum |ref|} (double), via `grid` partials.
cudaError_t launch_fbc_residual(const float* x1, const float* x0, const float* ref, float* r0, float* x1c, int rows,
                                int grid, double2* partial, double* out, cudaStream_t s);
// x += rest and the per-row sum-of-squares partials of the result.
cudaError_t launch_fbc_apply(float* x, const float* rest, float* ssp, int rows, cudaStream_t s);
// rest = xl - x1c.
cudaError_t launch_fbc_rest(const float* xl, const float* x1c, float* rest, int rows, int grid, cudaStream_t s);
// Classifier-free guidance: out = neg + g * (pos - neg), each operation rounded
// on its own (no FMA contraction).
cudaError_t launch_cfg_combine(const float* pos, const float* neg, float g, float* out, long long n, cudaStream_t s);
// In place bf16 -> fp16 for a weight tensor of n elements; values whose
// magnitude exceeds the fp16 range are counted into *overflow.
cudaError_t launch_bf16_to_f16(uint16_t* w, size_t n, unsigned int* overflow, cudaStream_t s);

// Test hook (operand ranges): *out = max(*out, max |a[i]|) over n fp16 values
// (n a multiple of 8, a 16-byte aligned); NaN counts as +inf.
cudaError_t launch_absmax_f16(const act_t* a, long long n, float* out, cudaStream_t s);

// Sets the calling thread's message returned by qi_last_error() (qidit.cu).
void set_last_error(const char* msg);

}  // namespace qi
