// Block-causal flash attention on the 5th-generation tensor cores (tcgen05).
//
// Mask (no mask tensor): query row with global index i attends to key j iff
//   (i < L and j <= i)  -- text rows are causal over text only
//   (i >= L and j < Lk) -- image rows see every text and image key.
// This is the port's "two SDPA calls" decomposition (text->text causal,
// image->all) done in one pass. Keys are visited in 128-row tiles from key 0 in
// the same order whatever the other query rows are, so an image row's result
// is the same in a joint pass and in an image-only pass over the stored text K/V.
//
// Work unit = 128 query rows of one head. A persistent grid (one CTA per SM)
// walks the units head-major, so the CTAs running at one time share a few heads'
// K/V in L2. Tensor memory (512 columns):
//   [0,128) O, [128,192) and [192,256) two Q slots (fp16 pairs, the A operand
//   of Q K^T), [256,384) S, [384,448) and [448,512) two P buffers (fp16 pairs,
//   the A operand of P V).
// Q sits in tensor memory, so Q K^T reads only K from shared memory (shared
// memory bandwidth, not the tensor core, is what a second operand stream from
// shared memory would saturate). P has buffers of its own, so S(j+1) only
// waits for the softmax warps to have read S(j) into registers, not for
// P(j) V(j): the Q K^T of the next tile runs under the softmax of this one.
//
// Two threads issue the MMAs: one Q K^T, one P V. A thread issuing an N = 128
// MMA is held about as long as the MMA runs, and each of its barrier checks
// leaves the tensor pipe idle, so with a single issuer the pipe ran dry between
// groups; with two, one thread's waits overlap the other's MMAs. P(j) V(j)
// waits for the softmax of tile j; the softmax writes P(j) once P(j-2) V(j-2)
// has read that buffer. Across units nothing drains: the next unit's Q is
// loaded into the other Q slot during the current unit, its Q K^T start as
// soon as S is read, and only its first P V waits for the epilogue to have read O.
//
// Roles (512 threads, four warpgroups):
//   warp 0      TMA producer of the K tiles (ring of 3); warp 2 of the V tiles
//   warp 1      TMEM owner and Q K^T issuer; warp 3 P V issuer (one thread each)
//   warps 4-11  softmax: warps 4-7 take keys 0-63 of every tile, warps 8-11
//               keys 64-127. A thread holds one query row's half tile (the TMEM
//               lane of its warp's quarter); the two halves of a row swap their maxima
//               through shared memory (a two-warp mbarrier), so both take the
//               tile's row maximum. The running max changes O only when it grows
//               by more than 2^8 (each half rescales its 64 O columns after the
//               previous P V has landed; the row sums use the same max, so the
//               result is unchanged). Each half writes its P columns and keeps
//               its own row sum.
//   warps 12-15 Q loader and epilogue: thread = query row. Loads the next unit's
//               Q rows into the free Q slot, then reads the finished unit's O,
//               releases it and stores O / (sum of the two row sums) as fp16 (or
//               MXFP8 codes and scales)
// The kernel launches at 128 registers a thread (four warps per SM sub-partition
// at 16 K registers each); after set-up the first warpgroup gives registers back
// (56) and the other three take them (152 each): 32 x (56 + 3 x 152) = 16 K per
// sub-partition, the launch's whole allotment.
// Every mbarrier wait is bounded; on expiry the error word is set, the roles
// leave their loops, the producers drain their loads and the issuers their MMAs
// before TMEM is released.
#include "internal.h"
#include "ptx.cuh"

namespace qi {
namespace {

constexpr int kBQ = 128;                       // query rows per unit
constexpr int kBKV = 128;                      // keys per tile
constexpr int kBox = 128 * 64 * 2;             // 128 rows x 64 dims: one 128-byte-swizzled TMA box (16 KB)
constexpr int kTile = 2 * kBox;                // K or V tile: 128 keys x 128 dims (32 KB)
constexpr int kStages = 3;                     // depth of the K ring and of the V ring
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColQ = 128;
constexpr uint32_t kColS = 256;
constexpr uint32_t kColP = 384;
constexpr uint32_t kIdescQK = idesc_f16_f32(128, kBKV);      // A = Q (tensor memory), B = K (K-major)
constexpr uint32_t kIdescPV = idesc_f16_f32_bmn(128, 128);   // A = P (tensor memory), B = V (MN-major)
constexpr float kRescaleLog2 = 8.0f;           // rescale O only when the max grows by > 2^8
constexpr int kThreads = 512;
constexpr uint32_t kRegsLow = 56;    // producers and MMA issuers
constexpr uint32_t kRegsHigh = 152;  // softmax halves and epilogue

// mbarriers
enum : int {
  kKFull = 0,
  kKEmpty = kKFull + kStages,
  kVFull = kKEmpty + kStages,
  kVEmpty = kVFull + kStages,
  kSFull = kVEmpty + kStages,  // S written
  kSFree = kSFull + 1,         // S read into registers (8 softmax warps)
  kPFull = kSFree + 1,         // [2] P buffer written (8 softmax warps)
  kPvDone = kPFull + 2,        // [2] P V of the buffer's tile complete
  kQFull = kPvDone + 2,        // [2] Q slot loaded (4 epilogue warps)
  kQEmpty = kQFull + 2,        // [2] last Q K^T of the slot's unit complete
  kOFull = kQEmpty + 2,        // unit's last P V complete
  kOEmpty = kOFull + 1,        // O read by the epilogue (4 epilogue warps)
  kLFull = kOEmpty + 1,        // [2] unit's row sums in shared memory (8 softmax warps)
  kXchg = kLFull + 2,          // [2][4] row-max swap of the two halves, per tile parity and quarter (2 warps)
  kDrainQK = kXchg + 8,
  kDrainPV = kDrainQK + 1,
  kNumBars = kDrainPV + 1
};
// shared memory after the K and V rings: barriers, TMEM address, abort flag,
// row sums [2 units][2 halves][128 rows], half-tile maxima [2 tiles][2 halves][128 rows]
constexpr int kSmem = 2 * kStages * kTile + 1024 + kNumBars * 8 + 16 + 2 * 2 * kBQ * 4 + 2 * 2 * kBQ * 4;

struct Unit {
  int head, r0, ntiles;
};

// Unit u: head u / nrt, query rows [r0, r0 + 128); key tiles to visit: image rows
// need all Lk keys, a unit of text rows only the keys up to its last row.
__device__ __forceinline__ Unit unit_of(const AttnParams& p, int u, int nrt) {
  Unit x;
  x.head = u / nrt;
  x.r0 = (u - x.head * nrt) * kBQ;
  const int last_q = p.q_off + min(x.r0 + kBQ, p.Rq) - 1;
  const int kend = last_q >= p.L ? p.Lk : min(p.Lk, last_q + 1);
  x.ntiles = (kend + kBKV - 1) / kBKV;
  return x;
}

__device__ __forceinline__ bool mbar_count4(int i) {
  return (i >= kQFull && i < kQFull + 2) || i == kOEmpty;
}
__device__ __forceinline__ bool mbar_count8(int i) {
  return i == kSFree || (i >= kPFull && i < kPFull + 2) || (i >= kLFull && i < kLFull + 2);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const AttnParams p,
            float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kStages * kTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kStages * kTile);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* lsum = reinterpret_cast<float*>(tmem_slot + 4);  // [2][2][kBQ]
  float* hmax = lsum + 2 * 2 * kBQ;                       // [2][2][kBQ]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nrt = (p.Rq + kBQ - 1) / kBQ;
  const int total = nrt * kHeads;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(&bars[i], mbar_count8(i) ? 8 : (mbar_count4(i) ? 4 : (i >= kXchg && i < kXchg + 8 ? 2 : 1)));
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
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

  // each role's code sits in the branch that set its register count
  if (warp < 4) {
    regs_release<kRegsLow>();
    if (lane != 0) {
      // one thread per warp works in this warpgroup
    } else if (warp == 0 || warp == 2) {
      // ---------------- TMA producers: warp 0 the K tiles, warp 2 the V tiles
      const bool is_k = warp == 0;
      uint64_t* full = bars + (is_k ? kKFull : kVFull);
      uint64_t* empty = bars + (is_k ? kKEmpty : kVEmpty);
      uint8_t* ring = is_k ? sK : sV;
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      uint32_t t = 0;  // tiles issued by this thread
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        const Unit un = unit_of(p, u, nrt);
        const int col0 = un.head * kHeadDim;
        for (int j = 0; j < un.ntiles; ++j) {
          const uint32_t st = t % kStages;
          if (*abort_flag || !mbar_wait(&empty[st], ((t / kStages) & 1u) ^ 1u)) {
            if (!*abort_flag) report_error(p.err, kErrTimeoutProducer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], kTile);
          tma_load_2d(ring + st * kTile, map, &full[st], col0, j * kBKV);
          tma_load_2d(ring + st * kTile + kBox, map, &full[st], col0 + 64, j * kBKV);
          ++t;
        }
      }
      // every load this thread issued must land before the CTA may exit
      for (uint32_t i = t > kStages ? t - kStages : 0; i < t; ++i)
        if (!mbar_wait(&full[i % kStages], (i / kStages) & 1u)) report_error(p.err, kErrTimeoutDrain);
    } else if (warp == 1) {
      // ---------------- Q K^T issuer: S(t) = Q K(t)^T, once the softmax warps have
      // read S(t - 1)
      // descriptor of stage 0's K tile; the others differ in the start address field
      const uint64_t kdesc0 = sw128_kmajor_desc(smem_u32(sK));
      uint32_t t = 0;
      int ku = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x, ++ku) {
        const Unit un = unit_of(p, u, nrt);
        const uint32_t qs = static_cast<uint32_t>(ku) & 1u;
        ok = !*abort_flag && mbar_wait(&bars[kQFull + qs], (static_cast<uint32_t>(ku) >> 1) & 1u);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tQ = tmem + kColQ + qs * 64;
        for (int j = 0; j < un.ntiles; ++j, ++t) {
          const uint32_t st = t % kStages;
          ok = (t < 1 || mbar_wait(&bars[kSFree], (t - 1) & 1u)) && mbar_wait(&bars[kKFull + st], (t / kStages) & 1u);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = kdesc0 + ((st * kTile) >> 4);
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k)
            mma_ts(tmem + kColS, tQ + k * 8, kd + (((k >> 2) * kBox + (k & 3) * 32) >> 4), kIdescQK,
                   k > 0 ? 1u : 0u);
          mma_commit(&bars[kSFull]);
          mma_commit(&bars[kKEmpty + st]);
        }
        if (!ok) break;
        // the Q slot is free once the unit's last Q K^T has completed
        mma_commit(&bars[kQEmpty + qs]);
      }
      if (!ok) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
      }
      mma_commit(&bars[kDrainQK]);
      if (!mbar_wait(&bars[kDrainQK], 0)) report_error(p.err, kErrTimeoutDrain);
    } else {
      // ---------------- P V issuer: O (+)= P(tt) V(tt); the first tile of a unit
      // overwrites O once the epilogue has read the previous unit's
      const uint64_t vdesc0 = sw128_mnmajor_desc(smem_u32(sV), kBox, 1024);
      uint32_t t = 0;
      int ku = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x, ++ku) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const Unit un = unit_of(p, u, nrt);
        for (int j = 0; j < un.ntiles; ++j, ++t) {
          const uint32_t b = t & 1u;
          const uint32_t st = t % kStages;
          ok = mbar_wait(&bars[kPFull + b], (t >> 1) & 1u) &&
               (j > 0 || ku == 0 || mbar_wait(&bars[kOEmpty], static_cast<uint32_t>(ku - 1) & 1u)) &&
               mbar_wait(&bars[kVFull + st], (t / kStages) & 1u);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd = vdesc0 + ((st * kTile) >> 4);
#pragma unroll
          for (int k = 0; k < kBKV / 16; ++k)
            // P columns: 16 keys = 8 columns of fp16 pairs; V rows: 16 keys = 2 KB
            mma_ts(tmem + kColO, tmem + kColP + b * 64 + k * 8, vd + ((k * 2048) >> 4), kIdescPV,
                   (j > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bars[kPvDone + b]);
          mma_commit(&bars[kVEmpty + st]);
        }
        if (!ok) break;
        mma_commit(&bars[kOFull]);
      }
      if (!ok && !*abort_flag) report_error(p.err, kErrTimeoutMma);
      if (!ok) *abort_flag = 1;
      mma_commit(&bars[kDrainPV]);
      if (!mbar_wait(&bars[kDrainPV], 0)) report_error(p.err, kErrTimeoutDrain);
    }
  } else if (warp < 12) {
    regs_acquire<kRegsHigh>();
    // ---------------- softmax: warps 4..7 keys 0-63, warps 8..11 keys 64-127 of every
    // tile; thread = one query row's half
    const int h = warp >= 8 ? 1 : 0;
    const int quarter = warp & 3;
    const int rit = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tO = tmem + lane_off + kColO + h * 64;  // this half's 64 O columns
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    uint32_t t = 0;
    int ku = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++ku) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const Unit un = unit_of(p, u, nrt);
      const int qg = p.q_off + un.r0 + rit;
      const int lim = qg < p.L ? qg + 1 : p.Lk;  // keys [0, lim) are visible
      float m_used = -INFINITY;
      float l = 0.f;
      for (int j = 0; j < un.ntiles; ++j) {
        const uint32_t tt = t + j;
        const uint32_t b = tt & 1u;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[kSFull], tt & 1u));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + kColS;
        // this half's 64 S columns: two loads in flight, one wait; then S may be
        // overwritten by the next tile's Q K^T
        uint32_t r[2][32];
        tmem_ld32(tS + h * 64, r[0]);
        tmem_ld32(tS + h * 64 + 32, r[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kSFree]);
        // keys at or past the row's limit become -inf (only tiles that reach a limit)
        const int kbase = j * kBKV + h * 64;
        if (__any_sync(0xffffffffu, kbase + 64 > lim)) {
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
          for (int i = 0; i < 32; i += 2)
            mx4[(i >> 1) & 3] = fmax3(mx4[(i >> 1) & 3], __uint_as_float(r[c][i]), __uint_as_float(r[c][i + 1]));
        // swap half maxima with the warp that holds the row's other half
        float* hm = hmax + (tt & 1u) * 2 * kBQ;
        hm[h * kBQ + rit] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        __syncwarp();
        uint64_t* xb = &bars[kXchg + (tt & 1u) * 4 + quarter];
        if (lane == 0) mbar_arrive(xb);
        ok = __all_sync(0xffffffffu, mbar_wait(xb, (tt >> 1) & 1u));
        if (!ok) break;
        tc_fence_after();
        // the tile's row maximum in base-2 units (scale > 0 keeps the order); the
        // same value in both halves
        const float mx = fmaxf(hm[rit], hm[kBQ + rit]) * scale_log2;
        const float m_new = fmaxf(m_used, mx);
        if (j == 0) {
          m_used = m_new;
        } else {
          // A row whose maximum grew by more than 2^8 brings O and its row sum to the
          // new maximum, once P V of the previous tile -- which may still be adding
          // into O -- is done. tcgen05.ld/st must be executed by the whole warp, so
          // the warp runs them if any row needs it; the other rows scale by exactly 1
          // and keep their maximum, so a row's result never depends on which rows
          // share its warp.
          const bool mine = m_new > m_used + kRescaleLog2;
          if (__any_sync(0xffffffffu, mine)) {
            const uint32_t tp = tt - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&bars[kPvDone + (tp & 1u)], (tp >> 1) & 1u))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float alpha = mine ? fast_exp2(m_used - m_new) : 1.0f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              uint32_t o[16];
              tmem_ld16(tO + c * 16, o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st16(tO + c * 16, o);
            }
            if (mine) {
              l *= alpha;
              m_used = m_new;
            }
          }
        }
        // P = 2^(s * scale - m) as fp16 pairs: this half's 64 keys go to columns
        // 32 h .. 32 h + 31 of P buffer tt % 2 (masked keys give 2^-inf = 0), once
        // P V of tile tt - 2 has read that buffer
        if (tt >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars[kPvDone + b], ((tt - 2) >> 1) & 1u));
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t tP = tmem + lane_off + kColP + b * 64;
        const uint64_t nm2 = f2_pack(-m_used, -m_used);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x2 =
                fma_f32x2(f2_pack(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1])), sc2, nm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const float e0 = fast_exp2(x0);
            const float e1 = fast_exp2(x1);
            rs2[i & 3] = add_f32x2(rs2[i & 3], f2_pack(e0, e1));
            pk[i] = pack_f16x2(e0, e1);
          }
          tmem_st16(tP + h * 32 + c * 16, pk);
        }
        float s[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) f2_unpack(rs2[i], s[2 * i], s[2 * i + 1]);
        l += ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
        tmem_st_wait();
        tc_fence_before();
        const bool last = j + 1 == un.ntiles;
        if (last) lsum[((ku & 1) * 2 + h) * kBQ + rit] = l;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[kPFull + b]);
          if (last) mbar_arrive(&bars[kLFull + (ku & 1)]);
        }
      }
      if (!ok) break;
      t += un.ntiles;
    }
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeoutEpilogue);
      *abort_flag = 1;
    }
  } else {
    regs_acquire<kRegsHigh>();
    // ---------------- Q loader and epilogue (warps 12..15), thread = one query row
    const int quarter = warp & 3;
    const int rit = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // Q rows of unit u (fp16, 128 dims = 64 columns of pairs) into Q slot `slot`;
    // rows past Rq are zero
    auto load_q = [&](int u, uint32_t slot) {
      const Unit un = unit_of(p, u, nrt);
      const int row = un.r0 + rit;
      const uint32_t dst = tmem + lane_off + kColQ + slot * 64;
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {
        uint32_t v[32];
        if (row < p.Rq) {
          const uint4* src =
              reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(row) * kHidden + un.head * kHeadDim) + hq * 8;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 w = src[i];
            v[i * 4 + 0] = w.x;
            v[i * 4 + 1] = w.y;
            v[i * 4 + 2] = w.z;
            v[i * 4 + 3] = w.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        tmem_st32(dst + hq * 32, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kQFull + slot]);
    };
    bool ok = true;
    int ku = 0;
    if (static_cast<int>(blockIdx.x) < total) load_q(blockIdx.x, 0);
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++ku) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      // the next unit's Q goes into the other slot once its previous unit's Q K^T are done
      const int un_next = u + static_cast<int>(gridDim.x);
      if (un_next < total) {
        const uint32_t ns = static_cast<uint32_t>(ku + 1) & 1u;
        if (ku + 1 >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars[kQEmpty + ns], (static_cast<uint32_t>(ku - 1) >> 1) & 1u));
          if (!ok) break;
        }
        load_q(un_next, ns);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[kOFull], static_cast<uint32_t>(ku) & 1u)) &&
           __all_sync(0xffffffffu, mbar_wait(&bars[kLFull + (ku & 1)], (static_cast<uint32_t>(ku) >> 1) & 1u));
      if (!ok) break;
      tc_fence_after();
      const Unit un = unit_of(p, u, nrt);
      const float l = lsum[((ku & 1) * 2) * kBQ + rit] + lsum[((ku & 1) * 2 + 1) * kBQ + rit];
      uint32_t o[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_off + kColO + c * 32, o[c]);
      tmem_ld_wait();
      // O is in registers: the next unit's first P V may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kOEmpty]);
      const int row = un.r0 + rit;
      if (row < p.Rq) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int col0 = un.head * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (p.oq) {
            // MXFP8: these 32 O columns are one block of the out-projection's A operand
            float ov[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __uint_as_float(o[c][i]) * inv;
            const int rg = p.oq_row0 + row;
            const int kcol = col0 + c * 32;
            p.osf[mx_sf_offset(rg, kcol / 32, p.oq_groups)] =
                mx_quant32(ov, p.oq + static_cast<size_t>(rg) * kHidden + kcol);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(p.o + static_cast<size_t>(row) * kHidden + col0 + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = pack_f16x2(__uint_as_float(o[c][8 * i + 0]) * inv, __uint_as_float(o[c][8 * i + 1]) * inv);
              w.y = pack_f16x2(__uint_as_float(o[c][8 * i + 2]) * inv, __uint_as_float(o[c][8 * i + 3]) * inv);
              w.z = pack_f16x2(__uint_as_float(o[c][8 * i + 4]) * inv, __uint_as_float(o[c][8 * i + 5]) * inv);
              w.w = pack_f16x2(__uint_as_float(o[c][8 * i + 6]) * inv, __uint_as_float(o[c][8 * i + 7]) * inv);
              d4[i] = w;
            }
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) report_error(p.err, kErrTimeoutEpilogue);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  if (p.Rq <= 0) return cudaSuccess;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = ensure_smem_limit(attn_tc, kSmem, attr_done);
  if (e != cudaSuccess) return e;
  // Q is read and O written with 16-byte vector accesses; K and V come by TMA
  if ((reinterpret_cast<uintptr_t>(p.q) & 15) != 0 || (reinterpret_cast<uintptr_t>(p.o) & 15) != 0)
    return cudaErrorInvalidValue;
  CUtensorMap mk, mv;
  if (!encode_map16(&mk, p.k, p.Lk, kHidden, kBKV, false) || !encode_map16(&mv, p.v, p.Lk, kHidden, kBKV, false))
    return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kHeadDim));
  const int units = ((p.Rq + kBQ - 1) / kBQ) * kHeads;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  const int grid = units < sms ? units : sms;
  return launch_dependent(attn_tc, dim3(grid), dim3(kThreads), kSmem, stream, mk, mv, p, scale_log2);
}

}  // namespace qi
