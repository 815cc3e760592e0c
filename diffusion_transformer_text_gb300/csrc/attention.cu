// Block-causal flash attention on the 5th-generation tensor cores (tcgen05).
//
// Mask (no mask tensor): query row with global index i attends to key j iff
//   (i < L and j <= i)  -- text rows are causal over text only
//   (i >= L and j < Lk) -- image rows see every text and image key.
// This is the port's "two SDPA calls" decomposition (text->text causal,
// image->all) done in one pass. Keys are visited in 128-row tiles from key 0 in
// the same order whatever the query tile holds, so an image row's result is the
// same in a joint pass and in an image-only pass over the stored text K/V.
//
// CTA = 128 query rows of one head; two CTAs share an SM (256 TMEM columns and
// ~98 KB of shared memory each), so one CTA's softmax overlaps the other's MMAs.
// Roles (192 threads):
//   warp 0     TMA producer: Q once, then K and V tiles (128 keys x 128 dims)
//   warp 1     TMEM owner and MMA issuer: S = Q K^T (M128 N128, both K-major),
//              then O += P V with P read from TMEM and V MN-major in shared memory
//   warps 2-5  softmax: thread = query row (TMEM lane). Reads its S row, keeps a
//              running max (O is rescaled only when the max grows by more than
//              2^8, the row sum uses the same max, so the result is unchanged),
//              writes P as fp16 over the S columns, and at the end scales O by
//              1 / rowsum and stores it.
// Every mbarrier wait is bounded; on expiry the error word is set and the CTA
// drains its copies and MMAs before releasing TMEM.
#include "internal.h"
#include "ptx.cuh"

namespace qi {
namespace {

constexpr int kBQ = 128;                       // query rows per CTA
constexpr int kBKV = 128;                      // keys per tile
constexpr int kHalfBytes = 128 * 64 * 2;       // one 128-row x 64-column swizzled box: 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;     // 128 rows x 128 dims: 32 KB
constexpr int kSmem = 3 * kTileBytes + 1024 + 256;
constexpr uint32_t kTmemCols = 256;            // S/P: columns [0,128), O: [128,256)
constexpr uint32_t kIdescQK = idesc_f16_f32(128, 128);
constexpr uint32_t kIdescPV = idesc_f16_f32_bmn(128, 128);
constexpr float kRescaleLog2 = 8.0f;           // rescale O only when the max grows by > 2^8

__global__ void __launch_bounds__(192, 2)
    attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, const AttnParams p, float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTileBytes;
  uint8_t* sV = smem + 2 * kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 3 * kTileBytes);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 2;
  uint64_t* v_full = bars + 3;
  uint64_t* v_empty = bars + 4;
  uint64_t* s_full = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* o_done = bars + 7;
  uint64_t* drain = bars + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int head = blockIdx.y;
  const int r0 = blockIdx.x * kBQ;
  const int col0 = head * kHeadDim;

  // keys this CTA visits: image rows need all Lk keys; a CTA of text rows only
  // needs keys up to its last row.
  const int last_q = p.q_off + min(r0 + kBQ, p.Rq) - 1;
  const int kend = last_q >= p.L ? p.Lk : min(p.Lk, last_q + 1);
  const int ntiles = (kend + kBKV - 1) / kBKV;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 9; ++i) mbar_init(&bars[i], i == 6 ? 4 : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;        // S (fp32) and, over its first 64 columns, P (fp16 pairs)
  const uint32_t tO = tmem + 128;  // O accumulator

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int k_last = -1, v_last = -1;  // last tile whose K / V load was issued
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(sQ, &tmQ, q_full, col0, r0);
      tma_load_2d(sQ + kHalfBytes, &tmQ, q_full, col0 + 64, r0);
      for (int j = 0; j < ntiles; ++j) {
        if (*abort_flag) break;
        const uint32_t par = j & 1;
        if (!mbar_wait(k_empty, par ^ 1u)) {
          report_error(p.err, kErrTimeoutProducer);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(k_full, kTileBytes);
        tma_load_2d(sK, &tmK, k_full, col0, j * kBKV);
        tma_load_2d(sK + kHalfBytes, &tmK, k_full, col0 + 64, j * kBKV);
        k_last = j;
        if (!mbar_wait(v_empty, par ^ 1u)) {
          report_error(p.err, kErrTimeoutProducer);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(v_full, kTileBytes);
        tma_load_2d(sV, &tmV, v_full, col0, j * kBKV);
        tma_load_2d(sV + kHalfBytes, &tmV, v_full, col0 + 64, j * kBKV);
        v_last = j;
      }
      // every load this thread issued must land before the CTA may exit
      if (!mbar_wait(q_full, 0)) report_error(p.err, kErrTimeoutDrain);
      if (k_last >= 0 && !mbar_wait(k_full, k_last & 1)) report_error(p.err, kErrTimeoutDrain);
      if (v_last >= 0 && !mbar_wait(v_full, v_last & 1)) report_error(p.err, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      bool ok = mbar_wait(q_full, 0);
      if (!ok) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
      }
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV);
      for (int j = 0; ok && j < ntiles; ++j) {
        if (*abort_flag) break;
        const uint32_t par = j & 1;
        // S may be overwritten once PV of the previous tile has read P
        if (j > 0 && !mbar_wait(o_done, par ^ 1u)) ok = false;
        if (ok && !mbar_wait(k_full, par)) ok = false;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {
          const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
          mma_ss(tS, sw128_kmajor_desc(q0 + off), sw128_kmajor_desc(k0 + off), kIdescQK, k > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        mma_commit(k_empty);
        if (!mbar_wait(p_full, par) || !mbar_wait(v_full, par)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kBKV / 16; ++k) {
          // P columns: 16 keys = 8 columns of fp16 pairs; V rows: 16 keys = 2 KB
          mma_ts(tO, tS + k * 8, sw128_mnmajor_desc(v0 + k * 2048, kHalfBytes, 1024), kIdescPV,
                      (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(v_empty);
      }
      if (!ok) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
      }
      mma_commit(drain);
      if (!mbar_wait(drain, 0)) report_error(p.err, kErrTimeoutDrain);
    }
  } else {
    // ---------------- softmax (warps 2..5), thread = one query row
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int row = r0 + row_in_tile;
    const int qg = p.q_off + row;
    const int lim = qg < p.L ? qg + 1 : p.Lk;  // keys [0, lim) are visible
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t par = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, par));
      if (!ok) break;
      tc_fence_after();
      const int kbase = j * kBKV;
      // the whole S row of this tile: four loads in flight, one wait
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, r[c]);
      tmem_ld_wait();
      // keys at or past the row's limit become -inf (only tiles that reach a limit)
      if (__any_sync(0xffffffffu, kbase + kBKV > lim)) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (kbase + c * 32 + i >= lim) r[c][i] = 0xff800000u;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(r[c][i]));
      // the tile's row maximum in base-2 units (scale > 0 keeps the order)
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
      const float m_new = fmaxf(m_used, mx);
      if (j == 0) {
        m_used = m_new;
      } else {
        // O holds the sum over earlier tiles (their PV finished before this S was
        // computed). A row whose maximum grew by more than 2^8 brings O and its
        // row sum to the new maximum. tcgen05.ld/st must be executed by the whole
        // warp, so the warp runs them if any row needs it; the other rows scale
        // by exactly 1 and keep their maximum, so a row's result never depends
        // on which rows share its warp.
        const bool mine = m_new > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, mine)) {
          const float alpha = mine ? fast_exp2(m_used - m_new) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t o[16];
            tmem_ld16(tO + lane_off + c * 16, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tO + lane_off + c * 16, o);
          }
          if (mine) {
            l *= alpha;
            m_used = m_new;
          }
        }
      }
      // P = 2^(s * scale - m) as fp16 pairs over the first 64 S columns (masked
      // keys give 2^-inf = 0). Chunk c of P covers S columns already read.
      float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = fast_exp2(fmaf(__uint_as_float(r[c][2 * i]), scale_log2, -m_used));
          const float b = fast_exp2(fmaf(__uint_as_float(r[c][2 * i + 1]), scale_log2, -m_used));
          rs4[i & 3] += a + b;
          pk[i] = pack_f16x2(a, b);
        }
        tmem_st16(tS + lane_off + c * 16, pk);
      }
      l += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // epilogue: wait for the last PV, O / l -> fp16
    if (ok && ntiles > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_done, (ntiles - 1) & 1));
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeoutEpilogue);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      act_t* dst = p.o + static_cast<size_t>(row) * kHidden + col0;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + lane_off + c * 32, r);
        tmem_ld_wait();
        if (row < p.Rq) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_f16x2(__uint_as_float(r[8 * i + 0]) * inv, __uint_as_float(r[8 * i + 1]) * inv);
            w.y = pack_f16x2(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv);
            w.z = pack_f16x2(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv);
            w.w = pack_f16x2(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv);
            d4[i] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  if (p.Rq <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap mq, mk, mv;
  if (!encode_map16(&mq, p.q, p.Rq, kHidden, 128, false) || !encode_map16(&mk, p.k, p.Lk, kHidden, 128, false) ||
      !encode_map16(&mv, p.v, p.Lk, kHidden, 128, false))
    return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kHeadDim));
  dim3 grid((p.Rq + kBQ - 1) / kBQ, kHeads);
  attn_tc<<<grid, 192, kSmem, stream>>>(mq, mk, mv, p, scale_log2);
  return cudaGetLastError();
}

}  // namespace qi
