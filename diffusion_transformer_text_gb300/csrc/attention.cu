// Block-causal flash attention for the single-stream DiT (first version,
// warp-level mma.sync m16n8k16 bf16 with fp32 accumulation).
//
// Mask (no mask tensor): query row with global index i attends to key j iff
//   (i < L and j <= i)  -- text rows are causal over text only
//   (i >= L and j < Lk) -- image rows see every text and image key.
// This is the port's "two SDPA calls" decomposition (text->text causal,
// image->all) done in one pass. Keys are visited in 64-row tiles from key 0 in
// the same order whatever the query tile holds, so an image row's result is the
// same in a joint pass and in an image-only pass over the stored text K/V.
//
// CTA: 128 query rows x one head (8 warps x 16 rows), K/V tiles of 64 keys
// double-buffered in shared memory with cp.async, online softmax in base 2.
#include "internal.h"
#include "ptx.cuh"

namespace qi {
namespace {

constexpr int kBQ = 128;
constexpr int kBKV = 64;
constexpr int kD = kHeadDim;  // 128
constexpr int kThreads = 256;
constexpr int kTileQBytes = kBQ * kD * 2;    // 32 KB
constexpr int kTileKVBytes = kBKV * kD * 2;  // 16 KB
constexpr int kSmem = kTileQBytes + 4 * kTileKVBytes;

// byte offset of element (row, col) in a [rows][128] bf16 tile whose 16-byte
// chunks are XOR-swizzled by (row & 7): conflict-free ldmatrix on 8 rows.
__device__ __forceinline__ uint32_t swz(int row, int col) {
  const int chunk = (col >> 3) ^ (row & 7);
  return static_cast<uint32_t>(row * (kD * 2) + chunk * 16 + (col & 7) * 2);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;  // n = 0 zero-fills the 16 bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Load a [rows][128] bf16 tile (row stride kHidden elements) into swizzled smem.
template <int ROWS>
__device__ __forceinline__ void load_tile(uint32_t sbase, const __nv_bfloat16* g, int row0, int nrows, int col0) {
  constexpr int kChunks = ROWS * (kD / 8);
#pragma unroll
  for (int i = 0; i < kChunks / kThreads; ++i) {
    const int c = threadIdx.x + i * kThreads;
    const int r = c >> 4;
    const int ch = c & 15;
    const bool ok = (row0 + r) < nrows;
    const __nv_bfloat16* src = g + (ok ? static_cast<size_t>(row0 + r) * kHidden + col0 + ch * 8 : 0);
    cp_async16(sbase + swz(r, ch * 8), src, ok);
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_fwd(const AttnParams p, float scale_log2) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + kTileQBytes;                 // 2 buffers
  const uint32_t sV = sK + 2 * kTileKVBytes;            // 2 buffers

  const int head = blockIdx.y;
  const int r0 = blockIdx.x * kBQ;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t4 = lane & 3;
  const int col0 = head * kD;

  // keys this CTA must visit
  const int last_q = p.q_off + min(r0 + kBQ, p.Rq) - 1;
  const int kend = last_q >= p.L ? p.Lk : min(p.Lk, last_q + 1);
  const int ntiles = (kend + kBKV - 1) / kBKV;

  load_tile<kBQ>(sQ, p.q, r0, p.Rq, col0);
  load_tile<kBKV>(sK, p.k, 0, kend, col0);
  load_tile<kBKV>(sV, p.v, 0, kend, col0);
  cp_async_commit();

  // the two query rows this thread holds: warp*16 + g and + 8
  const int qg0 = p.q_off + r0 + warp * 16 + g;
  const int qg1 = qg0 + 8;
  const int lim0 = qg0 < p.L ? qg0 + 1 : p.Lk;  // keys [0, lim) are visible
  const int lim1 = qg1 < p.L ? qg1 + 1 : p.Lk;

  uint32_t qf[8][4];
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const int mi = lane >> 3;  // which 8x8 matrix this lane addresses in ldmatrix.x4
  const int mr = lane & 7;

  for (int kt = 0; kt < ntiles; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < ntiles) {
      load_tile<kBKV>(sK + (buf ^ 1) * kTileKVBytes, p.k, (kt + 1) * kBKV, kend, col0);
      load_tile<kBKV>(sV + (buf ^ 1) * kTileKVBytes, p.v, (kt + 1) * kBKV, kend, col0);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    if (kt == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int row = warp * 16 + (mi & 1) * 8 + mr;
        const int col = kk * 16 + (mi >> 1) * 8;
        ldsm_x4(sQ + swz(row, col), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }

    // S = Q K^T for 64 keys: 8 n-blocks of 8 keys
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
    const uint32_t kb = sK + buf * kTileKVBytes;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int nb = 0; nb < 4; ++nb) {
        const int key = nb * 16 + (mi >> 1) * 8 + mr;
        const int col = kk * 16 + (mi & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + swz(key, col), b0, b1, b2, b3);
        mma16816(s[2 * nb], qf[kk], b0, b1);
        mma16816(s[2 * nb + 1], qf[kk], b2, b3);
      }
    }

    // scale, mask, online softmax (base 2)
    const int kbase = kt * kBKV;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kbase + nb * 8 + 2 * t4 + e;
        float a = s[nb][e] * scale_log2;
        float b = s[nb][2 + e] * scale_log2;
        a = key < lim0 ? a : -INFINITY;
        b = key < lim1 ? b : -INFINITY;
        s[nb][e] = a;
        s[nb][2 + e] = b;
        mx0 = fmaxf(mx0, a);
        mx1 = fmaxf(mx1, b);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0);
    const float mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float alpha0 = exp2f(m0 - base0);
    const float alpha1 = exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < 8; ++nb) {
      s[nb][0] = exp2f(s[nb][0] - base0);
      s[nb][1] = exp2f(s[nb][1] - base0);
      s[nb][2] = exp2f(s[nb][2] - base1);
      s[nb][3] = exp2f(s[nb][3] - base1);
      rs0 += s[nb][0] + s[nb][1];
      rs1 += s[nb][2] + s[nb][3];
    }
    l0 = l0 * alpha0 + rs0;
    l1 = l1 * alpha1 + rs1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= alpha0;
      o[i][1] *= alpha0;
      o[i][2] *= alpha1;
      o[i][3] *= alpha1;
    }

    // O += P V: 4 k-steps of 16 keys, 16 n-blocks of 8 dims
    const uint32_t vb = sV + buf * kTileKVBytes;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) {
        const int key = kk * 16 + (mi & 1) * 8 + mr;
        const int col = nd * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + swz(key, col), b0, b1, b2, b3);
        mma16816(o[2 * nd], pa, b0, b1);
        mma16816(o[2 * nd + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }

  // finish the row sums across the quad and write O
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int row0 = r0 + warp * 16 + g;
  const int row1 = row0 + 8;
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) {
    const int col = col0 + nd * 8 + 2 * t4;
    if (row0 < p.Rq)
      *reinterpret_cast<uint32_t*>(p.o + static_cast<size_t>(row0) * kHidden + col) =
          pack_bf16x2(o[nd][0] * inv0, o[nd][1] * inv0);
    if (row1 < p.Rq)
      *reinterpret_cast<uint32_t*>(p.o + static_cast<size_t>(row1) * kHidden + col) =
          pack_bf16x2(o[nd][2] * inv1, o[nd][3] * inv1);
  }
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  if (p.Rq <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kD));
  dim3 grid((p.Rq + kBQ - 1) / kBQ, kHeads);
  attn_fwd<<<grid, kThreads, kSmem, stream>>>(p, scale_log2);
  return cudaGetLastError();
}

}  // namespace qi
