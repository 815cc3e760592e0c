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
// K/V in L2. Each key tile's 128 keys are split in two halves, and each half
// keeps its own online softmax: its own running maximum, row sum and output
// accumulator O_h over the keys of that half of every tile. The two halves never
// wait for each other; the epilogue merges them (O = (O_0 a_0 + O_1 a_1) /
// (l_0 a_0 + l_1 a_1) with a_h = 2^(m_h - max(m_0, m_1))), as a split over keys
// is merged. Tensor memory (512 columns):
//   [0,128) O_0, [128,256) O_1, [256,384) S, [384,448) and [448,512) two P
//   buffers (fp16 pairs, the A operand of P V; half h at +32 h).
// Q sits in shared memory (a TMA tile, the A operand of Q K^T with K). P has
// buffers of its own, so S(j+1) only waits for the softmax warps to have read
// S(j) into registers, not for P(j) V(j).
//
// Two threads issue the MMAs: one Q K^T, one P V. A thread issuing an N = 128
// MMA is held about as long as the MMA runs, and each of its barrier checks
// leaves the tensor pipe idle, so with a single issuer the pipe ran dry between
// groups; with two, one thread's waits overlap the other's MMAs. P_h(j) V_h(j)
// (four MMAs into O_h) starts once half h has written P_h(j); half h writes
// P_h(j) once P_h(j-2) V_h(j-2) has read that buffer.
//
// Roles (512 threads, four warpgroups):
//   warp 0      TMA producer of the K tiles (ring of 3)
//   warp 1      TMEM owner and Q K^T issuer; warp 3 P V issuer (one thread each)
//   warp 2      TMA producer of the V tiles (ring of 2) and of each unit's Q tile,
//               once the previous unit's last Q K^T has completed
//   warps 4-11  softmax: warps 4-7 take keys 0-63 of every tile, warps 8-11
//               keys 64-127; thread = one query row's half (the TMEM lane of its
//               warp's quarter). A half's running max changes its O only when it
//               grows by more than 2^8 (rescaled after that half's previous P V has
//               landed; the row sum uses the same max, so the result is unchanged)
//   warps 12-15 epilogue: thread = query row; merges the two halves' O and row
//               sums and stores O as fp16 (or MXFP8 codes and scales)
// The kernel launches at 128 registers a thread (four warps per SM sub-partition
// at 16 K registers each); after set-up the first warpgroup and the epilogue give
// registers back (104 each) and the two softmax warpgroups take them (152 each):
// 32 x (104 + 2 x 152 + 104) = 16 K per sub-partition, the launch's whole allotment.
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
constexpr int kTile = 2 * kBox;                // Q, K or V tile: 128 rows x 128 dims (32 KB)
constexpr int kKStages = 3;                    // depth of the K ring
constexpr int kVStages = 2;                    // depth of the V ring
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;                  // O_h at kColO + 128 h
constexpr uint32_t kColS = 256;
constexpr uint32_t kColP = 384;                // buffer b at kColP + 64 b, half h at + 32 h
constexpr uint32_t kIdescQK = idesc_f16_f32(128, kBKV);      // A = Q, B = K (both K-major in shared memory)
constexpr uint32_t kIdescPV = idesc_f16_f32_bmn(128, 128);   // A = P (tensor memory), B = V (MN-major)
constexpr float kRescaleLog2 = 8.0f;           // rescale O_h only when its max grows by > 2^8
constexpr int kThreads = 512;
constexpr uint32_t kRegsLow = 104;   // producers and MMA issuers
constexpr uint32_t kRegsHigh = 152;  // softmax halves
constexpr uint32_t kRegsEpi = 104;   // epilogue
static_assert(kRegsLow + 2 * kRegsHigh + kRegsEpi == 4 * 128, "register split must equal the launch allotment");
// setmaxnreg.dec may only lower and setmaxnreg.inc only raise the launch's 128
static_assert(kRegsLow <= 128 && kRegsHigh >= 128 && kRegsEpi <= 128, "setmaxnreg direction");

// mbarriers
enum : int {
  kKFull = 0,
  kKEmpty = kKFull + kKStages,
  kVFull = kKEmpty + kKStages,
  kVEmpty = kVFull + kVStages,
  kQFull = kVEmpty + kVStages,  // unit's Q tile loaded
  kQEmpty = kQFull + 1,         // unit's last Q K^T complete
  kSFull = kQEmpty + 1,         // S written
  kSFree = kSFull + 1,          // S read into registers (8 softmax warps)
  kPFull = kSFree + 1,          // [buffer][half] P_h written (4 softmax warps)
  kPvDone = kPFull + 4,         // [buffer][half] P_h V_h of the buffer's tile complete
  kOFull = kPvDone + 4,         // unit's last P V complete
  kOEmpty = kOFull + 1,         // O_0 and O_1 read by the epilogue (4 epilogue warps)
  kLFull = kOEmpty + 1,         // unit's row sums and maxima in shared memory (8 softmax warps)
  kDrainQK = kLFull + 1,
  kDrainPV = kDrainQK + 1,
  kNumBars = kDrainPV + 1
};
__device__ __forceinline__ uint32_t bar_count(int i) {
  if (i == kSFree || i == kLFull) return 8;
  if ((i >= kPFull && i < kPFull + 4) || i == kOEmpty) return 4;
  return 1;
}
// shared memory: Q tile, K ring, V ring, barriers, TMEM address, abort flag,
// row sums and maxima [2 halves][128 rows] each
constexpr int kSmem = (1 + kKStages + kVStages) * kTile + 1024 + kNumBars * 8 + 16 + 2 * 2 * kBQ * 4;
static_assert(kSmem <= 227 * 1024, "shared memory over the per-block limit");

struct Unit {
  int head, r0, ntiles;
};

// 32 fp32 values as fp16 at dst (16-byte aligned): four 16-byte stores
__device__ __forceinline__ void store_o16(act_t* dst, const float (&v)[32]) {
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

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
            const __grid_constant__ CUtensorMap tmV, const AttnParams p, float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTile;
  uint8_t* sV = sK + kKStages * kTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kVStages * kTile);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* lsum = reinterpret_cast<float*>(tmem_slot + 4);  // [2][kBQ]
  float* msum = lsum + 2 * kBQ;                           // [2][kBQ]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nrt = (p.Rq + kBQ - 1) / kBQ;
  const int total = nrt * kHeads;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], bar_count(i));
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

  // each role's code sits in the branch that set its register count
  if (warp < 4) {
    regs_release<kRegsLow>();
    if (lane != 0) {
      // one thread per warp works in this warpgroup
    } else if (warp == 0) {
      // ---------------- TMA producer of the K tiles
      uint32_t t = 0;  // tiles issued
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        const Unit un = unit_of(p, u, nrt);
        const int col0 = un.head * kHeadDim;
        for (int j = 0; j < un.ntiles; ++j, ++t) {
          const uint32_t st = t % kKStages;
          if (*abort_flag || !mbar_wait(&bars[kKEmpty + st], ((t / kKStages) & 1u) ^ 1u)) {
            if (!*abort_flag) report_error(p.err, kErrTimeoutProducer);
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars[kKFull + st], kTile);
          tma_load_2d(sK + st * kTile, &tmK, &bars[kKFull + st], col0, j * kBKV);
          tma_load_2d(sK + st * kTile + kBox, &tmK, &bars[kKFull + st], col0 + 64, j * kBKV);
        }
      }
      // every load this thread issued must land before the CTA may exit
      for (uint32_t i = t > kKStages ? t - kKStages : 0; i < t; ++i)
        if (!mbar_wait(&bars[kKFull + i % kKStages], (i / kKStages) & 1u)) report_error(p.err, kErrTimeoutDrain);
    } else if (warp == 2) {
      // ---------------- TMA producer of the V tiles and of each unit's Q tile (once
      // the previous unit's last Q K^T has completed)
      uint32_t t = 0;  // V tiles issued
      int nq = 0;      // Q tiles issued
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
        const Unit un = unit_of(p, u, nrt);
        const int col0 = un.head * kHeadDim;
        if (*abort_flag || (nq > 0 && !mbar_wait(&bars[kQEmpty], static_cast<uint32_t>(nq - 1) & 1u))) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars[kQFull], kTile);
        tma_load_2d(sQ, &tmQ, &bars[kQFull], col0, un.r0);
        tma_load_2d(sQ + kBox, &tmQ, &bars[kQFull], col0 + 64, un.r0);
        ++nq;
        for (int j = 0; j < un.ntiles; ++j, ++t) {
          const uint32_t st = t % kVStages;
          if (*abort_flag || !mbar_wait(&bars[kVEmpty + st], ((t / kVStages) & 1u) ^ 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars[kVFull + st], kTile);
          tma_load_2d(sV + st * kTile, &tmV, &bars[kVFull + st], col0, j * kBKV);
          tma_load_2d(sV + st * kTile + kBox, &tmV, &bars[kVFull + st], col0 + 64, j * kBKV);
        }
      }
      if (!ok) {
        if (!*abort_flag) report_error(p.err, kErrTimeoutProducer);
        *abort_flag = 1;
      }
      for (uint32_t i = t > kVStages ? t - kVStages : 0; i < t; ++i)
        if (!mbar_wait(&bars[kVFull + i % kVStages], (i / kVStages) & 1u)) report_error(p.err, kErrTimeoutDrain);
      // the last Q load (a completed phase reads as complete until the barrier
      // moves on, and nothing else loads)
      if (nq > 0 && !mbar_wait(&bars[kQFull], static_cast<uint32_t>(nq - 1) & 1u))
        report_error(p.err, kErrTimeoutDrain);
    } else if (warp == 1) {
      // ---------------- Q K^T issuer: S(t) = Q K(t)^T, once the softmax warps have
      // read S(t - 1)
      const uint64_t qdesc = sw128_kmajor_desc(smem_u32(sQ));
      const uint64_t kdesc0 = sw128_kmajor_desc(smem_u32(sK));
      uint32_t t = 0;
      int ku = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total; u += gridDim.x, ++ku) {
        const Unit un = unit_of(p, u, nrt);
        ok = !*abort_flag && mbar_wait(&bars[kQFull], static_cast<uint32_t>(ku) & 1u);
        if (!ok) break;
        tc_fence_after();
        for (int j = 0; j < un.ntiles; ++j, ++t) {
          const uint32_t st = t % kKStages;
          ok = (t < 1 || mbar_wait(&bars[kSFree], (t - 1) & 1u)) &&
               mbar_wait(&bars[kKFull + st], (t / kKStages) & 1u);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd = kdesc0 + ((st * kTile) >> 4);
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t off = static_cast<uint32_t>(((k >> 2) * kBox + (k & 3) * 32) >> 4);
            mma_ss(tmem + kColS, qdesc + off, kd + off, kIdescQK, k > 0 ? 1u : 0u);
          }
          mma_commit(&bars[kSFull]);
          mma_commit(&bars[kKEmpty + st]);
        }
        if (!ok) break;
        // the Q tile is free once the unit's last Q K^T has completed
        mma_commit(&bars[kQEmpty]);
      }
      if (!ok) {
        report_error(p.err, kErrTimeoutMma);
        *abort_flag = 1;
      }
      mma_commit(&bars[kDrainQK]);
      if (!mbar_wait(&bars[kDrainQK], 0)) report_error(p.err, kErrTimeoutDrain);
    } else {
      // ---------------- P V issuer: O_h (+)= P_h(t) V_h(t) for each half h (keys 64 h
      // .. 64 h + 63 of the tile); the first tile of a unit overwrites O_0 and O_1
      // once the epilogue has read the previous unit's
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
          const uint32_t st = t % kVStages;
          ok = (j > 0 || ku == 0 || mbar_wait(&bars[kOEmpty], static_cast<uint32_t>(ku - 1) & 1u)) &&
               mbar_wait(&bars[kVFull + st], (t / kVStages) & 1u);
          if (!ok) break;
          const uint64_t vd = vdesc0 + ((st * kTile) >> 4);
          for (int h = 0; h < 2; ++h) {
            ok = mbar_wait(&bars[kPFull + b * 2 + h], (t >> 1) & 1u);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              // P columns: 16 keys = 8 columns of fp16 pairs; V rows: 16 keys = 2 KB
              mma_ts(tmem + kColO + 128u * h, tmem + kColP + b * 64 + h * 32 + k * 8,
                     vd + ((static_cast<uint32_t>(4 * h + k) * 2048) >> 4), kIdescPV, (j > 0 || k > 0) ? 1u : 0u);
            mma_commit(&bars[kPvDone + b * 2 + h]);
          }
          if (!ok) break;
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
    // tile; thread = one query row's half, with its own max, row sum and O_h
    const int h = warp >= 8 ? 1 : 0;
    const int quarter = warp & 3;
    const int rit = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tO = tmem + lane_off + kColO + 128u * h;
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
        // this half's 64 S columns: two loads in flight, one wait; then S may be
        // overwritten by the next tile's Q K^T
        uint32_t r[2][32];
        tmem_ld32(tmem + lane_off + kColS + h * 64, r[0]);
        tmem_ld32(tmem + lane_off + kColS + h * 64 + 32, r[1]);
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
        // this half's maximum in base-2 units (scale > 0 keeps the order)
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * scale_log2;
        const float m_new = fmaxf(m_used, mx);
        if (j == 0) {
          m_used = m_new;
        } else {
          // A row whose maximum grew by more than 2^8 brings O_h and its row sum to
          // the new maximum, once P_h V_h of the previous tile -- which may still be
          // adding into O_h -- is done. tcgen05.ld/st must be executed by the whole
          // warp, so the warp runs them if any row needs it; the other rows scale by
          // exactly 1 and keep their maximum, so a row's result never depends on which
          // rows share its warp. (A half whose keys so far were all masked has
          // m_used = -inf and O_h = 0: it takes the first finite maximum.)
          const bool mine = m_new > m_used + kRescaleLog2;
          if (__any_sync(0xffffffffu, mine)) {
            const uint32_t tp = tt - 1;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&bars[kPvDone + (tp & 1u) * 2 + h], (tp >> 1) & 1u))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float alpha = mine ? fast_exp2(m_used - m_new) : 1.0f;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
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
        // P_h = 2^(s * scale - m) as fp16 pairs (masked keys give 2^-inf = 0; a half
        // with no visible key yet subtracts 0 instead of -inf)
        const float base = m_used == -INFINITY ? 0.f : m_used;
        const uint64_t nm2 = f2_pack(-base, -base);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[2][16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x2 =
                fma_f32x2(f2_pack(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1])), sc2, nm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const float e0 = fast_exp2(x0);
            const float e1 = fast_exp2(x1);
            rs2[i & 3] = add_f32x2(rs2[i & 3], f2_pack(e0, e1));
            pk[c][i] = pack_f16x2(e0, e1);
          }
        }
        // P buffer b is free once P_h V_h of tile tt - 2 has read it
        if (tt >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars[kPvDone + b * 2 + h], ((tt - 2) >> 1) & 1u));
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t tP = tmem + lane_off + kColP + b * 64 + h * 32;
        tmem_st16(tP, pk[0]);
        tmem_st16(tP + 16, pk[1]);
        float s[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) f2_unpack(rs2[i], s[2 * i], s[2 * i + 1]);
        l += ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
        tmem_st_wait();
        tc_fence_before();
        const bool last = j + 1 == un.ntiles;
        if (last) {
          // the row sums' slots are free once the epilogue has read the previous
          // unit's (it cannot yet have read this unit's O, so the wait is for that phase)
          if (ku > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bars[kOEmpty], static_cast<uint32_t>(ku - 1) & 1u));
            if (!ok) break;
          }
          lsum[h * kBQ + rit] = l;
          msum[h * kBQ + rit] = m_used;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[kPFull + b * 2 + h]);
          if (last) mbar_arrive(&bars[kLFull]);
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
    regs_release<kRegsEpi>();
    // ---------------- epilogue (warps 12..15), thread = one query row: merges the
    // two halves and stores O
    const int quarter = warp & 3;
    const int rit = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    int ku = 0;
    for (int u = blockIdx.x; ok && u < total; u += gridDim.x, ++ku) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[kOFull], static_cast<uint32_t>(ku) & 1u)) &&
           __all_sync(0xffffffffu, mbar_wait(&bars[kLFull], static_cast<uint32_t>(ku) & 1u));
      if (!ok) break;
      tc_fence_after();
      const Unit un = unit_of(p, u, nrt);
      const float m0 = msum[rit], m1 = msum[kBQ + rit];
      // half 0 sees key 0 in the first tile, so m0 is finite; a half with no
      // visible key has m1 = -inf and weight 0
      const float mm = fmaxf(m0, m1);
      const float a0 = fast_exp2(m0 - mm);
      const float a1 = fast_exp2(m1 - mm);
      const float den = lsum[rit] * a0 + lsum[kBQ + rit] * a1;
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const float w0 = a0 * inv, w1 = a1 * inv;
      const int row = un.r0 + rit;
      const int col0 = un.head * kHeadDim;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + kColO + c * 32, o0);
        tmem_ld32(tmem + lane_off + kColO + 128 + c * 32, o1);
        tmem_ld_wait();
        if (c == 3) {
          // O_0 and O_1 are in registers: the next unit's first P V may overwrite them
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kOEmpty]);
        }
        if (row < p.Rq) {
          float ov[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __uint_as_float(o0[i]) * w0 + __uint_as_float(o1[i]) * w1;
          if (p.oq) {
            // MXFP8: these 32 O columns are one block of the out-projection's A operand
            const int rg = p.oq_row0 + row;
            const int kcol = col0 + c * 32;
            p.osf[mx_sf_offset(rg, kcol / 32, p.oq_groups)] =
                mx_quant32(ov, p.oq + static_cast<size_t>(rg) * kHidden + kcol);
          } else {
            store_o16(p.o + static_cast<size_t>(row) * kHidden + col0 + c * 32, ov);
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
  CUtensorMap mq, mk, mv;
  if (!encode_map16(&mq, p.q, p.Rq, kHidden, kBQ, false) || !encode_map16(&mk, p.k, p.Lk, kHidden, kBKV, false) ||
      !encode_map16(&mv, p.v, p.Lk, kHidden, kBKV, false))
    return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kHeadDim));
  const int units = ((p.Rq + kBQ - 1) / kBQ) * kHeads;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  const int grid = units < sms ? units : sms;
  return launch_dependent(attn_tc, dim3(grid), dim3(kThreads), kSmem, stream, mq, mk, mv, p, scale_log2);
}

}  // namespace qi
