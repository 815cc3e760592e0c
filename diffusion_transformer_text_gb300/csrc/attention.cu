// Block-causal flash attention on the 5th-generation tensor cores (tcgen05).
//
// Mask (no mask tensor): query row with global index i attends to key j iff
//   (i < L and j <= i)  -- text rows are causal over text only
//   (i >= L and j < Lk) -- image rows see every text and image key.
// This is the port's "two SDPA calls" decomposition (text->text causal,
// image->all) done in one pass. Keys are visited in 64-row tiles from key 0 in
// the same order whatever the query tile holds, so an image row's result is the
// same in a joint pass and in an image-only pass over the stored text K/V.
//
// CTA = 128 query rows of one head; two CTAs share an SM (256 TMEM columns and
// ~98 KB of shared memory each). Keys come in 64-row tiles and S is double
// buffered in tensor memory, so the MMA warp computes S(j+1) = Q K(j+1)^T while
// the softmax warps turn S(j) into P(j):
//   TMEM columns [0,64) S buffer 0, [64,128) S buffer 1, [128,256) O.
// Roles (224 threads):
//   warp 0     TMA producer of Q (once) and the K tiles (64 keys x 128 dims, two
//              slots); warp 6 produces the V tiles (two slots). Separate threads,
//              so a K load never queues behind a V slot that PV still reads.
//   warp 1     TMEM owner and MMA issuer, in the order S(0), S(1), PV(0), S(2),
//              PV(1), ...: S(j+1) = Q K^T (M128 N64, both K-major) once PV(j-1)
//              has read the P that shared its buffer; O += P(j) V(j) with P read
//              from TMEM and V MN-major in shared memory
//   warps 2-5  softmax: thread = query row (TMEM lane). Reads its S row, keeps a
//              running max (O is rescaled only when the max grows by more than
//              2^8 -- after the previous PV has landed -- and the row sum uses the
//              same max, so the result is unchanged), writes P as fp16 over the
//              first 32 columns of the S buffer, and at the end scales O by
//              1 / rowsum and stores it.
// Every mbarrier wait is bounded; on expiry the error word is set and the CTA
// drains its copies and MMAs before releasing TMEM.
#include "internal.h"
#include "ptx.cuh"

namespace qi {
namespace {

constexpr int kBQ = 128;                       // query rows per CTA
constexpr int kBKV = 64;                       // keys per tile
constexpr int kQHalf = 128 * 64 * 2;           // Q: 128 rows x 64 dims, one swizzled box (16 KB)
constexpr int kQBytes = 2 * kQHalf;            // Q: 128 rows x 128 dims (32 KB)
constexpr int kKVHalf = kBKV * 64 * 2;         // K or V: 64 rows x 64 dims (8 KB)
constexpr int kKVBytes = 2 * kKVHalf;          // K or V tile: 64 rows x 128 dims (16 KB)
constexpr int kSmem = kQBytes + 4 * kKVBytes + 1024 + 256;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kOCol = 128;
constexpr uint32_t kIdescQK = idesc_f16_f32(128, kBKV);
constexpr uint32_t kIdescPV = idesc_f16_f32_bmn(128, 128);
constexpr float kRescaleLog2 = 8.0f;           // rescale O only when the max grows by > 2^8

constexpr int kThreads = 224;

__global__ void __launch_bounds__(kThreads, 2)
    attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, const AttnParams p, float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kQBytes;                 // two slots
  uint8_t* sV = sK + 2 * kKVBytes;              // two slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + 2 * kKVBytes);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* k_empty = bars + 3;   // [2]
  uint64_t* v_full = bars + 5;    // [2]
  uint64_t* v_empty = bars + 7;   // [2]
  uint64_t* s_full = bars + 9;    // [2]
  uint64_t* p_full = bars + 11;   // [2], one arrival per softmax warp
  uint64_t* pv_done = bars + 13;  // one phase per tile
  uint64_t* drain = bars + 14;
  constexpr int kBars = 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBars);
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
    for (int i = 0; i < kBars; ++i) mbar_init(&bars[i], (i == 11 || i == 12) ? 4 : 1);
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
  // the set-up above may overlap the previous kernel; every activation read and
  // write comes after this wait
  grid_dep_wait();
  grid_dep_launch_dependents();
  const uint32_t tO = tmem + kOCol;

  if (warp == 0 || warp == 6) {
    if (lane == 0) {
      // ---------------- TMA producers: warp 0 Q and K, warp 6 V
      const bool is_k = warp == 0;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* dst = is_k ? sK : sV;
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      int last[2] = {-1, -1};  // last tile whose load was issued, per slot
      if (is_k) {
        mbar_arrive_expect_tx(q_full, kQBytes);
        tma_load_2d(sQ, &tmQ, q_full, col0, r0);
        tma_load_2d(sQ + kQHalf, &tmQ, q_full, col0 + 64, r0);
      }
      for (int j = 0; j < ntiles; ++j) {
        if (*abort_flag) break;
        const int slot = j & 1;
        if (!mbar_wait(&empty[slot], ((j >> 1) & 1) ^ 1u)) {
          report_error(p.err, kErrTimeoutProducer);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[slot], kKVBytes);
        tma_load_2d(dst + slot * kKVBytes, map, &full[slot], col0, j * kBKV);
        tma_load_2d(dst + slot * kKVBytes + kKVHalf, map, &full[slot], col0 + 64, j * kBKV);
        last[slot] = j;
      }
      // every load this thread issued must land before the CTA may exit
      if (is_k && !mbar_wait(q_full, 0)) report_error(p.err, kErrTimeoutDrain);
      for (int s2 = 0; s2 < 2; ++s2)
        if (last[s2] >= 0 && !mbar_wait(&full[s2], (last[s2] >> 1) & 1)) report_error(p.err, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      bool ok = mbar_wait(q_full, 0);
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV);
      // S(j) = Q K(j)^T into S buffer j % 2
      auto issue_qk = [&](int j) -> bool {
        const int slot = j & 1;
        if (!mbar_wait(&k_full[slot], (j >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t kb = k0 + slot * kKVBytes;
        const uint32_t tS = tmem + static_cast<uint32_t>(slot * kBKV);
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {
          const uint32_t qoff = (k >> 2) * kQHalf + (k & 3) * 32;
          const uint32_t koff = (k >> 2) * kKVHalf + (k & 3) * 32;
          mma_ss(tS, sw128_kmajor_desc(q0 + qoff), sw128_kmajor_desc(kb + koff), kIdescQK, k > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[slot]);
        mma_commit(&k_empty[slot]);
        return true;
      };
      if (ok && ntiles > 0) ok = issue_qk(0);
      for (int j = 0; ok && j < ntiles; ++j) {
        if (*abort_flag) break;
        const int slot = j & 1;
        if (j + 1 < ntiles) {
          // S buffer (j+1) % 2 held P(j-1): PV(j-1) must have read it
          if (j >= 1 && !mbar_wait(pv_done, (j - 1) & 1)) {
            ok = false;
            break;
          }
          if (!issue_qk(j + 1)) {
            ok = false;
            break;
          }
        }
        if (!mbar_wait(&p_full[slot], (j >> 1) & 1) || !mbar_wait(&v_full[slot], (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tP = tmem + static_cast<uint32_t>(slot * kBKV);
        const uint32_t vb = v0 + slot * kKVBytes;
#pragma unroll
        for (int k = 0; k < kBKV / 16; ++k) {
          // P columns: 16 keys = 8 columns of fp16 pairs; V rows: 16 keys = 2 KB
          mma_ts(tO, tP + k * 8, sw128_mnmajor_desc(vb + k * 2048, kKVHalf, 1024), kIdescPV,
                 (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(pv_done);
        mma_commit(&v_empty[slot]);
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
      const int slot = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[slot], (j >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(slot * kBKV);
      const int kbase = j * kBKV;
      // the whole S row of this tile: two loads in flight, one wait
      uint32_t r[2][32];
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(tS + c * 32, r[c]);
      tmem_ld_wait();
      // keys at or past the row's limit become -inf (only tiles that reach a limit)
      if (__any_sync(0xffffffffu, kbase + kBKV > lim)) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (kbase + c * 32 + i >= lim) r[c][i] = 0xff800000u;
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(r[c][i]));
      // the tile's row maximum in base-2 units (scale > 0 keeps the order)
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
      const float m_new = fmaxf(m_used, mx);
      if (j == 0) {
        m_used = m_new;
      } else {
        // A row whose maximum grew by more than 2^8 brings O and its row sum to the
        // new maximum, once PV(j-1) -- which may still be adding into O -- is done.
        // tcgen05.ld/st must be executed by the whole warp, so the warp runs them if
        // any row needs it; the other rows scale by exactly 1 and keep their
        // maximum, so a row's result never depends on which rows share its warp.
        const bool mine = m_new > m_used + kRescaleLog2;
        if (__any_sync(0xffffffffu, mine)) {
          if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
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
      // P = 2^(s * scale - m) as fp16 pairs over the first 32 columns of the S
      // buffer (masked keys give 2^-inf = 0); those columns were read above.
      float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = fast_exp2(fmaf(__uint_as_float(r[c][2 * i]), scale_log2, -m_used));
          const float b = fast_exp2(fmaf(__uint_as_float(r[c][2 * i + 1]), scale_log2, -m_used));
          rs4[i & 3] += a + b;
          pk[i] = pack_f16x2(a, b);
        }
        tmem_st16(tS + c * 16, pk);
      }
      l += (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[slot]);
    }
    // epilogue: O / l -> fp16 once every MMA has completed. With S double-buffered,
    // PV(n-2) may still be running when the last softmax ends, so a parity wait on
    // pv_done could match phase n-3; the MMA warp's single-use drain barrier
    // (committed after its last MMA) cannot.
    if (ok && ntiles > 0) ok = __all_sync(0xffffffffu, mbar_wait(drain, 0));
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
        if (row < p.Rq && p.oq) {
          // MXFP8: these 32 O columns are one block of the out-projection's A operand
          float ov[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __uint_as_float(r[i]) * inv;
          const int rg = p.oq_row0 + row;
          const int kcol = col0 + c * 32;
          p.osf[mx_sf_offset(rg, kcol / 32, p.oq_groups)] =
              mx_quant32(ov, p.oq + static_cast<size_t>(rg) * kHidden + kcol);
        } else if (row < p.Rq) {
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
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_limit(attn_tc, kSmem, attr_done);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv;
  if (!encode_map16(&mq, p.q, p.Rq, kHidden, kBQ, false) || !encode_map16(&mk, p.k, p.Lk, kHidden, kBKV, false) ||
      !encode_map16(&mv, p.v, p.Lk, kHidden, kBKV, false))
    return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kHeadDim));
  dim3 grid((p.Rq + kBQ - 1) / kBQ, kHeads);
  return launch_dependent(attn_tc, grid, dim3(kThreads), kSmem, stream, mq, mk, mv, p, scale_log2);
}

}  // namespace qi
