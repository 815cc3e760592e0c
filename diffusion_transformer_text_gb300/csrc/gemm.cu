// Persistent, warp-specialised tcgen05 GEMM for the DiT block's dense
// contractions (QKV, out-projection, SwiGLU gate/up, down, text projection),
// with the block's elementwise work fused into the epilogue.
//
// D[M, N] = A[M, K] * B[N, K]^T; A = fp16 activations, B = fp16 weights (converted
// from the bf16 checkpoint values; [out, in] row-major), fp32 accumulation in
// tensor memory. The plain fp32 epilogue (a test hook) takes bf16 operands.
//
// MXFP8 kernel (gemm_mx_tc): A and B are E4M3 bytes with one UE8M0 scale per 32
// values along K, stored in 512-byte chunks (128 rows x 4 scales, byte
// (r % 32) * 16 + ((r % 128) / 32) * 4 + k) ordered [K / 128][rows / 128]. A
// stage then covers K = 128; its scale chunks arrive by bulk copy with the
// tiles, are copied into a per-stage set of TMEM columns (tcgen05.cp) and feed
// four block-scaled MMAs (K = 32 each, the scale byte chosen per MMA). The two
// 256-column accumulators fill tensor memory, so a tile keeps its scales in the
// first 64 columns of the other accumulator: written only after the previous
// tile's MMAs have completed and its epilogue has read those columns.
//
// Two kernels share the epilogues. The fp16 / bf16 GEMMs run on CTA pairs
// (gemm_pair_tc: a cluster of two CTAs computes 256 x 256 tiles with
// tcgen05.mma.cta_group::2, each CTA loading its 128 A rows and half of the B
// rows); the MXFP8 GEMM runs one CTA per 128 x 256 tile (gemm_mx_tc).
//
// Roles per CTA (192 threads):
//   warp 0     TMA producer: A and B tiles into a ring of stages (pair: 128x64
//              fp16 A and 128x64 fp16 B, 6 stages; MXFP8: 128x128 E4M3 A, 256x128
//              E4M3 B and the scale chunks, 4 stages)
//   warp 1     TMEM owner and MMA issuer (one thread; the pair's leader only):
//              4 x tcgen05.mma per stage (pair: M = 256, K = 16 each; MXFP8:
//              M = 128, K = 32 each), accumulating into one of two 256-column
//              TMEM buffers
//   warps 2-5  epilogue: each thread owns one accumulator row (TMEM lane),
//              reads 32 columns at a time and applies the fused epilogue while
//              the MMA warp fills the other TMEM buffer.
//
// Every GEMM row is computed the same way whatever M is (no split-K, fixed
// K order), so a row's result does not depend on the other rows in the pass:
// this is what makes the text K/V of a joint pass equal a text-only pass.
//
// Last wave: when the tiles left after the full waves fill at most half the
// grid (of CTAs, or of pairs), each of them runs as two 128-column halves (the
// MMA with N = 128 produces the same bits per element as with N = 256), so the
// last wave takes half as long (the gate/up weight's 64-row interleave makes a
// 128-column half hold matching gate and up columns).
#include "internal.h"
#include "ptx.cuh"

namespace qi {
namespace {

constexpr int kMxStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kEpiScratch = 4 * 32 * 33 * 4;  // per epilogue warp: one 32 x 32 fp32 chunk, stride 33
constexpr int kSfChunk = 512;                  // MXFP8 scales of 128 rows x 128 K

// MXFP8 kernel geometry: 128-byte tile rows as for 16-bit operands, so a stage
// packs K = 128 E4M3 values and adds the scale chunks of A (one) and B (two).
struct MxGeo {
  static constexpr int kSF = 3 * kSfChunk;
  static constexpr int kStage = kABytes + kBBytes + kSF;
  static constexpr int kK = 128;  // K elements per stage
  static constexpr int kAcc = 2;  // TMEM accumulators (256 columns each)
  static constexpr int kSmem = kMxStages * kStage + 1024 + 256 + kEpiScratch;
};
// MXFP8: a tile's stage-s scales sit at columns 16 s (A: +0..3, B: +4..11) of the OTHER
// accumulator, i.e. inside the tile the epilogue is draining.
constexpr uint32_t kTmemCols = 512;  // two 256-column accumulators
constexpr int kGroupN = 8;           // tiles sweep 8 column tiles per row tile for L2 reuse

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& mt, int& nt) {
  const int group = kGroupN * num_m;
  const int g = t / group;
  const int first_n = g * kGroupN;
  const int gsz = min(kGroupN, num_n - first_n);
  const int local = t - g * group;
  mt = local / gsz;
  nt = first_n + local % gsz;
}

// Work unit u: a whole tile for u < tail_start, else half h of tile
// tail_start + (u - tail_start) / 2 (columns 128 h .. 128 h + 127).
__device__ __forceinline__ void unit_tile(int u, int tail_start, int& tile, int& half) {
  if (u < tail_start) {
    tile = u;
    half = -1;
  } else {
    tile = tail_start + ((u - tail_start) >> 1);
    half = (u - tail_start) & 1;
  }
}

__device__ __forceinline__ float row_rinv(const float* ssp, int row) {
  const float4* p = reinterpret_cast<const float4*>(ssp + static_cast<size_t>(row) * kSspParts);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kSspParts / 4; ++i) {
    const float4 v = p[i];
    s += v.x;
    s += v.y;
    s += v.z;
    s += v.w;
  }
  return rsqrtf(s * (1.0f / kHidden) + kEps);
}

__device__ __forceinline__ void store_f16x32(act_t* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w;
    w.x = pack_f16x2(v[8 * i + 0], v[8 * i + 1]);
    w.y = pack_f16x2(v[8 * i + 2], v[8 * i + 3]);
    w.z = pack_f16x2(v[8 * i + 4], v[8 * i + 5]);
    w.w = pack_f16x2(v[8 * i + 6], v[8 * i + 7]);
    d[i] = w;
  }
}

// ---------------------------------------------------------------- epilogues

// MXFP8: the next tile's scale sets go into the first 64 columns of the
// accumulator this epilogue drains; once every epilogue warp has read them
// (chunks 0 and 1 of 32 columns) the warp tells the MMA issuer.
__device__ __forceinline__ void release_sf_cols(uint64_t* sf_bar, int c) {
  if (sf_bar == nullptr || c != 1) return;
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(sf_bar);
}

// The same release right after the warp has read columns 0..63 into registers
// (the QKV and SwiGLU epilogues read them first, so the MMA issuer can start the
// next tile's scale copies before the rest of the epilogue runs).
__device__ __forceinline__ void release_sf_now(uint64_t* sf_bar) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(sf_bar);
}

template <bool EARLY>
__device__ __forceinline__ void epi_qkv(const GemmParams& p, uint32_t taddr, int row, int n0, int ncols,
                                        uint64_t* sf_bar) {
  const bool valid = row < p.M;
  float rinv = 0.f;
  const float* cs = nullptr;
  const float* sn = nullptr;
  act_t* dst = nullptr;
  const int section = n0 / kHidden;  // 0 Q, 1 K, 2 V
  const int col_in = n0 - section * kHidden;
  if (valid) {
    rinv = row_rinv(p.ssp_in, row);
    const bool second = p.split_row > 0 && row >= p.split_row;  // second prompt's image rows
    const int r = second ? row - p.split_row : row;
    const bool text = r < p.n_text;
    const size_t trow = text ? static_cast<size_t>(r) : static_cast<size_t>(r - p.n_text);
    cs = (text ? p.txt_cos : (second ? p.img_cos2 : p.img_cos)) + trow * kRopeCols;
    sn = (text ? p.txt_sin : (second ? p.img_sin2 : p.img_sin)) + trow * kRopeCols;
    if (section == 0)
      dst = p.q + static_cast<size_t>(row) * kHidden + col_in;
    else if (second)
      dst = (section == 1 ? p.k2 : p.v2) + static_cast<size_t>(r + p.kv_row_off2) * kHidden + col_in;
    else
      dst = (section == 1 ? p.k : p.v) + static_cast<size_t>(row + p.kv_row_off) * kHidden + col_in;
  }
  auto chunk = [&](int c, const uint32_t(&r)[32]) {
    if (!valid) return;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * rinv;
    if (section < 2) {
      // interleaved rotary: pair j = columns (2j, 2j+1) of the head, angle column j
      const int j0 = ((col_in + c * 32) & (kHeadDim - 1)) >> 1;
      float cv[16], sv[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 a = reinterpret_cast<const float4*>(cs + j0)[i];
        const float4 b = reinterpret_cast<const float4*>(sn + j0)[i];
        cv[4 * i] = a.x; cv[4 * i + 1] = a.y; cv[4 * i + 2] = a.z; cv[4 * i + 3] = a.w;
        sv[4 * i] = b.x; sv[4 * i + 1] = b.y; sv[4 * i + 2] = b.z; sv[4 * i + 3] = b.w;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float a = v[2 * j], b = v[2 * j + 1];
        v[2 * j] = a * cv[j] - b * sv[j];
        v[2 * j + 1] = a * sv[j] + b * cv[j];
      }
    }
    store_f16x32(dst + c * 32, v);
  };
  int c0 = 0;
  if (EARLY) {
    // MXFP8: columns 0..63 hold the next tile's scale sets once released
    uint32_t r0[32], r1[32];
    tmem_ld32(taddr, r0);
    tmem_ld32(taddr + 32, r1);
    tmem_ld_wait();
    release_sf_now(sf_bar);
    chunk(0, r0);
    chunk(1, r1);
    c0 = 2;
  }
#pragma unroll 1
  for (int c = c0; c < ncols / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    tmem_ld_wait();
    if (!EARLY) release_sf_cols(sf_bar, c);
    chunk(c, r);
  }
}

// Residual epilogue. The accumulator arrives one row per lane; each 32 x 32
// chunk is transposed through shared memory (stride 33: conflict-free both
// ways) so that lane i handles column i of the warp's 32 rows and every global
// access of the fp32 residual and the fp16 copy is one contiguous row segment.
// Per row: x = acc + bias (set) or x += gate * acc; xa = fp16(x * (1 + scale));
// the row's sum of squares over each 128 columns is accumulated per lane and
// reduced per row in a fixed order.
__device__ __forceinline__ void epi_resid(const GemmParams& p, uint32_t taddr, int row0, int lane, int n0, int ncols,
                                          float* sm, uint64_t* sf_bar) {
  float sq[32];
#pragma unroll
  for (int rr = 0; rr < 32; ++rr) sq[rr] = 0.f;
  const bool own_row = !p.resid_set && row0 + lane < p.M;
#pragma unroll 1
  for (int c = 0; c < ncols / 32; ++c) {
    // the next chunk's residual segment of this lane's row (one 128-byte line) into L1
    if (own_row && c + 1 < ncols / 32)
      prefetch_l1(p.x + static_cast<size_t>(row0 + lane) * kHidden + n0 + (c + 1) * 32);
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    tmem_ld_wait();
    release_sf_cols(sf_bar, c);
#pragma unroll
    for (int k = 0; k < 32; ++k) sm[lane * 33 + k] = __uint_as_float(r[k]);
    __syncwarp();
    float acc[32];
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) acc[rr] = sm[rr * 33 + lane];
    __syncwarp();
    const int col = n0 + c * 32 + lane;
    const float g_img = p.mod[p.gate_chunk * kHidden + col];
    const float g_txt = p.mod[kMod + p.gate_chunk * kHidden + col];
    const float s_img = 1.f + p.mod[p.scale_chunk * kHidden + col];
    const float s_txt = 1.f + p.mod[kMod + p.scale_chunk * kHidden + col];
    const float bias = p.resid_set ? bf16_bits_to_float(p.bias[col]) : 0.f;
    // all 32 residual loads in flight before any store (the stores could alias
    // them as far as the compiler knows, which would serialise the rows)
    float xo[32];
    const float* xcol = p.x + static_cast<size_t>(row0) * kHidden + col;
#pragma unroll
    for (int rr = 0; rr < 32; ++rr)
      xo[rr] = (!p.resid_set && row0 + rr < p.M) ? xcol[static_cast<size_t>(rr) * kHidden] : 0.f;
#pragma unroll
    for (int rr = 0; rr < 32; ++rr) {
      const int row = row0 + rr;
      if (row < p.M) {
        const bool txt = row < p.n_text;
        const size_t idx = static_cast<size_t>(row) * kHidden + col;
        const float xn = p.resid_set ? acc[rr] + bias : xo[rr] + (txt ? g_txt : g_img) * acc[rr];
        p.x[idx] = xn;
        sq[rr] += xn * xn;
        p.xa[idx] = __float2half_rn(xn * (txt ? s_txt : s_img));
      }
    }
    if ((c & 3) == 3) {
      // end of a 128-column partial: per-row sums through shared memory, fixed order
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) sm[rr * 33 + lane] = sq[rr];
      __syncwarp();
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) ss += sm[lane * 33 + k];
      __syncwarp();
      if (row0 + lane < p.M) p.ssp_out[static_cast<size_t>(row0 + lane) * kSspParts + n0 / kSspCols + c / 4] = ss;
#pragma unroll
      for (int rr = 0; rr < 32; ++rr) sq[rr] = 0.f;
    }
  }
}

// SwiGLU epilogue. The gate/up weight is interleaved in 64-row groups, so every
// 128 tile columns hold the gate rows of 64 hidden units followed by their up
// rows: block b = n0 / 128 + j of the tile yields h columns 64 b .. 64 b + 63,
// and a 128-column half tile is a whole block.
template <bool EARLY>
__device__ __forceinline__ void epi_swiglu(const GemmParams& p, uint32_t taddr, int row, int n0, int ncols,
                                           uint64_t* sf_bar) {
  const bool valid = row < p.M;
  const float rinv = valid ? row_rinv(p.ssp_in, row) : 0.f;
  auto chunk = [&](int j, int c, const uint32_t(&g)[32], const uint32_t(&u)[32]) {
    if (!valid) return;
    float hv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float a = __uint_as_float(g[i]) * rinv;
      const float b = __uint_as_float(u[i]) * rinv;
      // silu(a) = a / (1 + e^-a) with the fast division: its few-ulp error is far
      // below the fp16 / E4M3 rounding of h (and e^-a = inf gives -0, the limit)
      hv[i] = __fdividef(a, 1.f + __expf(-a)) * b;
    }
    const int hcol = (n0 / 128 + j) * 64 + c * 32;
    if (p.hq) {
      // MXFP8: these 32 h columns are one block of the down GEMM's A operand
      p.hsf[mx_sf_offset(row, hcol / 32, (p.M + kBM - 1) / kBM)] =
          mx_quant32(hv, p.hq + static_cast<size_t>(row) * kFfn + hcol);
    } else {
      store_f16x32(p.h + static_cast<size_t>(row) * kFfn + hcol, hv);
    }
  };
  int j0 = 0;
  if (EARLY) {
    // MXFP8: gate columns 0..63 hold the next tile's scale sets once released
    uint32_t g0[32], g1[32];
    tmem_ld32(taddr, g0);
    tmem_ld32(taddr + 32, g1);
    tmem_ld_wait();
    release_sf_now(sf_bar);
    {
      uint32_t u[32];
      tmem_ld32(taddr + 64, u);
      tmem_ld_wait();
      chunk(0, 0, g0, u);
    }
    {
      uint32_t u[32];
      tmem_ld32(taddr + 96, u);
      tmem_ld_wait();
      chunk(0, 1, g1, u);
    }
    j0 = 1;
  }
#pragma unroll 1
  for (int j = j0; j < ncols / 128; ++j) {
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      uint32_t g[32], u[32];
      tmem_ld32(taddr + j * 128 + c * 32, g);
      tmem_ld32(taddr + j * 128 + 64 + c * 32, u);
      tmem_ld_wait();
      if (!EARLY) release_sf_cols(sf_bar, 2 * j + c);
      chunk(j, c, g, u);
    }
  }
}

__device__ __forceinline__ void epi_f32(const GemmParams& p, uint32_t taddr, int row, int n0, int ncols,
                                        uint64_t* sf_bar) {
  const bool valid = row < p.M;
  float* dst = p.d + static_cast<size_t>(row) * p.N + n0;
#pragma unroll 1
  for (int c = 0; c < ncols / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(taddr + c * 32, r);
    tmem_ld_wait();
    release_sf_cols(sf_bar, c);
    if (!valid) continue;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      reinterpret_cast<float4*>(dst + c * 32)[i] =
          make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                      __uint_as_float(r[4 * i + 3]));
  }
}

// ---------------------------------------------------------------- kernel

template <int KIND>
__global__ void __launch_bounds__(192, 1)
    gemm_mx_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const GemmParams p) {
  using G = MxGeo;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kMxStages * kABytes;
  uint8_t* sSF = sB + kMxStages * kBBytes;  // MXFP8 scale chunks, G::kSF bytes per stage
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kMxStages * G::kStage);
  uint64_t* empty = full + kMxStages;
  uint64_t* tfull = empty + kMxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* sffree = drain + 1;  // MXFP8: scale columns of accumulator a readable again
  uint64_t* never = sffree + 2;  // test hook: nothing ever arrives here
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (p.M + kBM - 1) / kBM;
  const int num_n = p.N / kBN;
  const int tiles = num_m * num_n;
  const int total = p.tail_start + 2 * (tiles - p.tail_start);  // work units
  const int kblocks = p.K / G::kK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
      mbar_init(&sffree[a], 4);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above may overlap the previous kernel; every activation read and
  // write comes after this wait
  grid_dep_wait();
  grid_dep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        if (*abort_flag) break;
        int tile, half, mt, nt;
        unit_tile(t, p.tail_start, tile, half);
        tile_coords(tile, num_m, num_n, mt, nt);
        // a half tile still loads a 256-row B box (rows past N read as zero) and uses its first 128 rows
        const int n_row = nt * kBN + (half > 0 ? kBN / 2 : 0);
        const int sfb_chunks = half >= 0 ? 1 : 2;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u)) {
            report_error(p.err, kErrTimeoutProducer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], G::kStage - (2 - sfb_chunks) * kSfChunk);
          tma_load_2d(sA + stage * kABytes, &tmA, &full[stage], kb * G::kK, mt * kBM);
          tma_load_2d(sB + stage * kBBytes, &tmB, &full[stage], kb * G::kK, n_row);
          uint8_t* sf = sSF + stage * G::kSF;
          bulk_load(sf, p.sfa + (static_cast<size_t>(kb) * num_m + mt) * kSfChunk, kSfChunk, &full[stage]);
          bulk_load(sf + kSfChunk, p.sfb + (static_cast<size_t>(kb) * (p.N / 128) + n_row / 128) * kSfChunk,
                    sfb_chunks * kSfChunk, &full[stage]);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every load this thread issued must land before the CTA may exit
      for (int s = 0; s < kMxStages; ++s)
        if ((issued_mask >> s) & 1u)
          if (!mbar_wait(&full[s], (issued_parity >> s) & 1u)) report_error(p.err, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      if (p.stall_test && !mbar_wait(never, 0)) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
        ok = false;
      }
      int local = 0;  // tiles this CTA has issued
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++local) {
        if (*abort_flag) break;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u)) {
          report_error(p.err, kErrTimeoutMma);
          *abort_flag = 1;
          break;
        }
        if (local > 0) {
          // the previous tile (other accumulator) must be complete, and its epilogue
          // past the first 64 columns, before this tile's scales go there
          const uint32_t prev_parity = static_cast<uint32_t>((local - 1) >> 1) & 1u;
          if (!mbar_wait(&tfull[acc ^ 1u], prev_parity) || !mbar_wait(&sffree[acc ^ 1u], prev_parity)) {
            report_error(p.err, kErrTimeoutMma);
            *abort_flag = 1;
            break;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        int tile_u, half_u;
        unit_tile(t, p.tail_start, tile_u, half_u);
        const int n_mma = half_u >= 0 ? kBN / 2 : kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase)) {
            report_error(p.err, kErrTimeoutMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kABytes);
          const uint32_t b0 = smem_u32(sB + stage * kBBytes);
          // this stage's scale set: the MMAs that last read it (kMxStages stages ago)
          // completed before the producer could refill the stage
          const uint32_t sf_t = tmem_base + (acc ^ 1u) * kBN + 16 * stage;
          const uint32_t sf_s = smem_u32(sSF + stage * G::kSF);
          tmem_cp_sf(sf_t, plain_rows16_desc(sf_s));
          tmem_cp_sf(sf_t + 4, plain_rows16_desc(sf_s + kSfChunk));
          if (half_u < 0) tmem_cp_sf(sf_t + 8, plain_rows16_desc(sf_s + 2 * kSfChunk));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_mxf8(d, sw128_kmajor_desc(a0 + 32 * k), sw128_kmajor_desc(b0 + 32 * k),
                     idesc_mxf8_f32(kBM, n_mma, static_cast<uint32_t>(k)), sf_t, sf_t + 4, (kb | k) != 0 ? 1u : 0u);
          mma_commit(&empty[stage]);
          if (++stage == kMxStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        if (++acc == G::kAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs of this thread must finish before TMEM is released
      mma_commit(drain);
      if (!mbar_wait(drain, 0)) report_error(p.err, kErrTimeoutDrain);
    }
  } else {
    // ---------------- epilogue (warps 2..5)
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = quarter * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      int tile, half, mt, nt;
      unit_tile(t, p.tail_start, tile, half);
      tile_coords(tile, num_m, num_n, mt, nt);
      const int n0 = nt * kBN + (half > 0 ? kBN / 2 : 0);
      const int ncols = half >= 0 ? kBN / 2 : kBN;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase));
      if (!ok) {
        if (lane == 0) report_error(p.err, kErrTimeoutEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN;
      const int row = mt * kBM + row_in_tile;
      uint64_t* sf_bar = &sffree[acc];
      if (KIND == kEpiQkv)
        epi_qkv<true>(p, taddr, row, n0, ncols, sf_bar);
      else if (KIND == kEpiResid)
        epi_resid(p, taddr, mt * kBM + quarter * 32, lane, n0, ncols,
                  reinterpret_cast<float*>(smem + kMxStages * G::kStage + 256) + (warp - 2) * 32 * 33, sf_bar);
      else if (KIND == kEpiSwiglu)
        epi_swiglu<true>(p, taddr, row, n0, ncols, sf_bar);
      else
        epi_f32(p, taddr, row, n0, ncols, sf_bar);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == G::kAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- CTA-pair kernel
//
// fp16 / bf16 operands: a cluster of two CTAs computes 256 x 256 tiles with
// tcgen05.mma.cta_group::2. Each CTA loads its own 128 A rows and half of the
// tile's 256 B rows (16 KB + 16 KB per stage, 6 stages); both CTAs' loads count
// on the leader's `full` barrier; the leader's single MMA thread issues
// M = 256 MMAs and its commits arrive on the barriers of both CTAs (stage free,
// accumulator full, drain). Each CTA's epilogue warps drain their own 128
// accumulator rows and arrive on the leader's `tempty` barrier (4 warps x 2).
// Per SM this halves the B bytes loaded and read by the tensor core per MMA.
constexpr int kPairStages = 6;
constexpr int kPairB = (kBN / 2) * kBK * 2;     // 16 KB: this CTA's half of the B tile
constexpr int kPairStage = kABytes + kPairB;    // 32 KB
constexpr int kPairSmem = kPairStages * kPairStage + 1024 + 256 + kEpiScratch;
constexpr int kPairRows = 2 * kBM;              // rows of a pair tile

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    gemm_pair_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the same offsets in both CTAs: the pair's MMA addresses the peer's operands by them
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPairStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStage);  // leader's are used
  uint64_t* empty = full + kPairStages;
  uint64_t* tfull = empty + kPairStages;
  uint64_t* tempty = tfull + 2;  // leader's are used
  uint64_t* drain = tempty + 2;
  uint64_t* never = drain + 1;   // test hook: nothing ever arrives here
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int num_m = (p.M + kPairRows - 1) / kPairRows;
  const int num_n = p.N / kBN;
  const int tiles = num_m * num_n;
  const int total = p.tail_start + 2 * (tiles - p.tail_start);  // work units
  const int kblocks = p.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above may overlap the previous kernel; every activation read and
  // write comes after this wait
  grid_dep_wait();
  grid_dep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs): own A rows and own half of B
      const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // leader: stages whose expect_tx it posted
      bool ok = true;
      for (int t = pair; ok && t < total; t += npairs) {
        if (*abort_flag) break;
        int tile, half, mt, nt;
        unit_tile(t, p.tail_start, tile, half);
        tile_coords(tile, num_m, num_n, mt, nt);
        const int a_row = mt * kPairRows + static_cast<int>(rank) * kBM;
        // a half tile (N = 128) takes 64 B rows from each CTA; the 128-row box's
        // other rows are loaded but not read
        const int b_rows = half >= 0 ? kBN / 4 : kBN / 2;
        const int b_row = nt * kBN + (half > 0 ? kBN / 2 : 0) + static_cast<int>(rank) * b_rows;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u)) {
            report_error(p.err, kErrTimeoutProducer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (rank == 0) {
            mbar_arrive_expect_tx(&full[stage], 2 * kPairStage);
            issued_mask |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
          tma_load_2d_pair(sA + stage * kABytes, &tmA, full_leader + 8u * stage, kb * kBK, a_row);
          tma_load_2d_pair(sB + stage * kPairB, &tmB, full_leader + 8u * stage, kb * kBK, b_row);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the leader's posted stages must complete (both CTAs' bytes) before the pair may exit
      if (rank == 0)
        for (int s = 0; s < kPairStages; ++s)
          if ((issued_mask >> s) & 1u)
            if (!mbar_wait(&full[s], (issued_parity >> s) & 1u)) report_error(p.err, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (leader only)
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      if (p.stall_test && !mbar_wait(never, 0)) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
        ok = false;
      }
      for (int t = pair; ok && t < total; t += npairs) {
        if (*abort_flag) break;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u)) {
          report_error(p.err, kErrTimeoutMma);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        int tile_u, half_u;
        unit_tile(t, p.tail_start, tile_u, half_u);
        const int n_mma = half_u >= 0 ? kBN / 2 : kBN;
        const uint32_t idesc =
            KIND == kEpiF32 ? idesc_bf16_f32(kPairRows, n_mma) : idesc_f16_f32(kPairRows, n_mma);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase)) {
            report_error(p.err, kErrTimeoutMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * kABytes);
          const uint32_t b0 = smem_u32(sB + stage * kPairB);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_ss_pair(d, sw128_kmajor_desc(a0 + 32 * k), sw128_kmajor_desc(b0 + 32 * k), idesc,
                        (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair(&empty[stage]);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // arrives in both CTAs once every MMA above has completed
      mma_commit_pair(drain);
    }
  } else {
    // ---------------- epilogue (warps 2..5 of both CTAs): this CTA's 128 rows
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = static_cast<int>(rank) * kBM + quarter * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
    uint32_t acc = 0, acc_phase = 0;
    for (int t = pair; t < total; t += npairs) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      int tile, half, mt, nt;
      unit_tile(t, p.tail_start, tile, half);
      tile_coords(tile, num_m, num_n, mt, nt);
      const int n0 = nt * kBN + (half > 0 ? kBN / 2 : 0);
      const int ncols = half >= 0 ? kBN / 2 : kBN;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase));
      if (!ok) {
        if (lane == 0) report_error(p.err, kErrTimeoutEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN;
      const int row = mt * kPairRows + row_in_tile;
      if (KIND == kEpiQkv)
        epi_qkv<false>(p, taddr, row, n0, ncols, nullptr);
      else if (KIND == kEpiResid)
        epi_resid(p, taddr, row - lane, lane, n0, ncols,
                  reinterpret_cast<float*>(smem + kPairStages * kPairStage + 256) + (warp - 2) * 32 * 33, nullptr);
      else if (KIND == kEpiSwiglu)
        epi_swiglu<false>(p, taddr, row, n0, ncols, nullptr);
      else
        epi_f32(p, taddr, row, n0, ncols, nullptr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // all MMAs done (they read both CTAs' shared memory and write both TMEMs)
  if (warp == 1 && lane == 0 && !mbar_wait(drain, 0)) report_error(p.err, kErrTimeoutDrain);
  __syncwarp();
  __syncthreads();
  if (rank != 0 && threadIdx.x == 0 && *abort_flag) {
    // after an abort the peer's last loads may not have been consumed by the
    // leader's MMAs; they land within microseconds (their barrier is the leader's)
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the other may still touch its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int KIND>
cudaError_t launch_pair_kind(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, int grid,
                             cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_limit(gemm_pair_tc<KIND>, kPairSmem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_dependent(gemm_pair_tc<KIND>, dim3(grid), dim3(192), kPairSmem, stream, a, b, p);
}

cudaError_t launch_pair_any(EpiKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                            int grid_ctas, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  if (p.N % kBN != 0 || p.K % kBK != 0) return cudaErrorInvalidValue;
  const int clusters = grid_ctas / 2;
  if (clusters < 1) return cudaErrorInvalidValue;
  const int tiles = ((p.M + kPairRows - 1) / kPairRows) * (p.N / kBN);
  // split the last wave's tiles into 128-column halves when they fill at most half the pairs
  GemmParams q = p;
  q.tail_start = tiles;
  const int rem = tiles % clusters;
  if (rem > 0 && 2 * rem <= clusters) q.tail_start = tiles - rem;
  const int units = q.tail_start + 2 * (tiles - q.tail_start);
  const int grid = 2 * (units < clusters ? units : clusters);
  switch (kind) {
    case kEpiQkv:
      return launch_pair_kind<kEpiQkv>(a, b, q, grid, stream);
    case kEpiResid:
      return launch_pair_kind<kEpiResid>(a, b, q, grid, stream);
    case kEpiSwiglu:
      return launch_pair_kind<kEpiSwiglu>(a, b, q, grid, stream);
    case kEpiF32:
      return launch_pair_kind<kEpiF32>(a, b, q, grid, stream);
  }
  return cudaErrorInvalidValue;
}

template <int KIND>
cudaError_t launch_mx_kind(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, int grid,
                           cudaStream_t stream) {
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_limit(gemm_mx_tc<KIND>, MxGeo::kSmem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_dependent(gemm_mx_tc<KIND>, dim3(grid), dim3(192), MxGeo::kSmem, stream, a, b, p);
}

cudaError_t launch_mx_any(EpiKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                          int grid_ctas, cudaStream_t stream) {
  if (p.M <= 0) return cudaSuccess;
  if (p.N % kBN != 0 || p.K % MxGeo::kK != 0) return cudaErrorInvalidValue;
  if (p.sfa == nullptr || p.sfb == nullptr) return cudaErrorInvalidValue;
  const int tiles = ((p.M + kBM - 1) / kBM) * (p.N / kBN);
  // split the last wave's tiles into 128-column halves when they fill at most half the grid
  GemmParams q = p;
  q.tail_start = tiles;
  const int rem = tiles % grid_ctas;
  if (rem > 0 && 2 * rem <= grid_ctas) q.tail_start = tiles - rem;
  const int units = q.tail_start + 2 * (tiles - q.tail_start);
  const int grid = units < grid_ctas ? units : grid_ctas;
  switch (kind) {
    case kEpiQkv:
      return launch_mx_kind<kEpiQkv>(a, b, q, grid, stream);
    case kEpiResid:
      return launch_mx_kind<kEpiResid>(a, b, q, grid, stream);
    case kEpiSwiglu:
      return launch_mx_kind<kEpiSwiglu>(a, b, q, grid, stream);
    case kEpiF32:
      return launch_mx_kind<kEpiF32>(a, b, q, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(EpiKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                        int grid_ctas, cudaStream_t stream) {
  return launch_pair_any(kind, a, b, p, grid_ctas, stream);
}

cudaError_t launch_gemm_mx(EpiKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                           int grid_ctas, cudaStream_t stream) {
  return launch_mx_any(kind, a, b, p, grid_ctas, stream);
}

}  // namespace qi
