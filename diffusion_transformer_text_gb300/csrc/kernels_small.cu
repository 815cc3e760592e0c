// The DiT step's small, memory-bound kernels: timestep embedding and the
// shared modulation (GEMVs over 2 rows), text pre-norm, image-token projection,
// output head, RoPE tables, noise packing and the Euler update.
#include <math.h>

#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace qi {
namespace {

__device__ __forceinline__ float silu(float a) { return a / (1.f + expf(-a)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- timestep

// e[0] = sinusoid of 1000*t, e[1] = sinusoid of 0; [cos(1000 t w_k) | sin(...)],
// w_k = 10000^(-k/128), k < 128.
__global__ void timestep_embed_kernel(float t, float* e) {
  const int k = threadIdx.x;  // 0..127
  const float w = powf(10000.f, -static_cast<float>(k) / 128.f);
  const float a = (1000.f * t) * w;
  e[k] = cosf(a);
  e[128 + k] = sinf(a);
  e[256 + k] = 1.f;  // cos(0)
  e[256 + 128 + k] = 0.f;
}

// y[r][o] = W[o] . act(x[r]) + b[o] for r = 0, 1; act = silu or identity.
// Each warp computes kOutPerWarp outputs at a time; W rows are read once, 16 bytes
// per lane. The grid is a multiple of the SM count and output group g goes to
// block g % gridDim.x, so every SM streams the same share of W (a grid of whole
// 32-output blocks left some SMs a quarter more than others); the first chunk of
// a warp's rows is requested before x is staged in shared memory.
constexpr int kOutPerWarp = 4;
__global__ void __launch_bounds__(256) gemv2_kernel(const float* __restrict__ x, int in_dim,
                                                    const uint16_t* __restrict__ W, const uint16_t* __restrict__ b,
                                                    int out_dim, float* __restrict__ y, int silu_in) {
  extern __shared__ float xs[];  // [2][in_dim]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int groups = (out_dim + kOutPerWarp - 1) / kOutPerWarp;
  const int chunks = in_dim / 8;
  int grp = blockIdx.x + warp * gridDim.x;
  const uint4* wr[kOutPerWarp];
  auto rows_of = [&](int gi) {
#pragma unroll
    for (int j = 0; j < kOutPerWarp; ++j)
      wr[j] = reinterpret_cast<const uint4*>(W + static_cast<size_t>(min(gi * kOutPerWarp + j, out_dim - 1)) * in_dim);
  };
  uint4 wv[kOutPerWarp];
  if (grp < groups) {
    rows_of(grp);
    if (lane < chunks) {
#pragma unroll
      for (int j = 0; j < kOutPerWarp; ++j) wv[j] = wr[j][lane];
    }
  }
  for (int i = threadIdx.x; i < 2 * in_dim; i += blockDim.x) {
    const float v = x[i];
    xs[i] = silu_in ? silu(v) : v;
  }
  __syncthreads();
  for (; grp < groups; grp += warps_total) {
    const int o_base = grp * kOutPerWarp;
    // the warp's rows side by side, so each lane has a 16-byte load of every row in
    // flight; each row's per-lane sum runs over c in the same order as alone
    float a0[kOutPerWarp], a1[kOutPerWarp];
#pragma unroll
    for (int j = 0; j < kOutPerWarp; ++j) a0[j] = a1[j] = 0.f;
    for (int c = lane; c < chunks; c += 32) {
      if (c != lane) {
#pragma unroll
        for (int j = 0; j < kOutPerWarp; ++j) wv[j] = wr[j][c];
      }
      const float* x0 = xs + c * 8;
      const float* x1 = xs + in_dim + c * 8;
#pragma unroll
      for (int j = 0; j < kOutPerWarp; ++j) {
        const uint32_t ws[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __uint_as_float(ws[q] << 16);
          const float hi = __uint_as_float(ws[q] & 0xFFFF0000u);
          a0[j] += lo * x0[2 * q] + hi * x0[2 * q + 1];
          a1[j] += lo * x1[2 * q] + hi * x1[2 * q + 1];
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kOutPerWarp; ++j) {
      const int o = o_base + j;
      const float s0 = warp_sum(a0[j]);
      const float s1 = warp_sum(a1[j]);
      if (lane == 0 && o < out_dim) {
        const float bb = bf16_bits_to_float(b[o]);
        y[o] = s0 + bb;
        y[out_dim + o] = s1 + bb;
      }
    }
    // the next group's first chunk
    if (grp + warps_total < groups) {
      rows_of(grp + warps_total);
      if (lane < chunks) {
#pragma unroll
        for (int j = 0; j < kOutPerWarp; ++j) wv[j] = wr[j][lane];
      }
    }
  }
}

// The same product for 4096-wide rows, streamed. One CTA per SM takes a
// contiguous range of W rows (8 KB each); a producer warp bulk-copies them into a
// ring of kGvStages stages of kGvRows rows, so every SM keeps ~192 KB of its share
// of W in flight (per-warp loads left too little in flight to reach the copy
// rate). Eight consumer warps never wait for one another: thread t holds act(x) at
// elements 8 t .. 8 t + 7 and 2048 + 8 t .. 2048 + 8 t + 7 of both rows in
// registers and multiplies the same elements of every W row; each warp sums its
// lanes' products of a stage (a butterfly that leaves one of the stage's 8 sums
// on each group of 4 lanes), parks them in shared memory and releases the stage.
// At the end the 8 warps' sums of every output are added in warp order, so an
// output is summed the same way on every call.
constexpr int kGvIn = 4096;
constexpr int kGvRows = 4;                                  // W rows per stage
constexpr int kGvStageBytes = kGvRows * kGvIn * 2;         // 32 KB
constexpr int kGvStages = 6;
constexpr int kGvWarps = 8;                                 // consumer warps
constexpr int kGvThreads = 32 * (kGvWarps + 1);             // + the producer warp
constexpr int kGvMaxRows = 128;                             // W rows per CTA at most
constexpr int kGvSmem = kGvStages * kGvStageBytes + 2 * kGvStages * 8 + kGvWarps * kGvMaxRows * 2 * 4 + 16;

__global__ void __launch_bounds__(kGvThreads, 1)
    gemv_stream_kernel(const float* __restrict__ x, const uint16_t* __restrict__ W, const uint16_t* __restrict__ b,
                       int out_dim, float* __restrict__ y, int silu_in, int* err) {
  extern __shared__ __align__(128) uint8_t gv_smem[];
  uint8_t* ring = gv_smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(gv_smem + kGvStages * kGvStageBytes);
  uint64_t* empty = full + kGvStages;
  float* part = reinterpret_cast<float*>(empty + kGvStages);  // [warp][row][2]
  volatile int* failed = reinterpret_cast<volatile int*>(part + kGvWarps * kGvMaxRows * 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r_begin = static_cast<int>(static_cast<long long>(out_dim) * blockIdx.x / gridDim.x);
  const int r_end = static_cast<int>(static_cast<long long>(out_dim) * (blockIdx.x + 1) / gridDim.x);
  const int nrows = r_end - r_begin;  // <= kGvMaxRows (the launcher's grid)
  const int ngroups = (nrows + kGvRows - 1) / kGvRows;
  if (tid == 0) {
    for (int i = 0; i < kGvStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGvWarps);
    }
    *failed = 0;
    fence_barrier_init();
  }
  __syncthreads();
  grid_dep_launch_dependents();
  // Launched dependent on the previous kernel (a step's timestep and modulation
  // GEMVs), the W stream starts at once: the weights are written only by copies
  // when they are loaded. x is read, and y written, after the previous kernel.
  if (warp == kGvWarps) {
    // ---------------- producer: group gi into stage gi % kGvStages once every
    // consumer warp has released the stage's previous group
    if (lane == 0) {
      int gi = 0;
      for (; gi < ngroups; ++gi) {
        const int st = gi % kGvStages;
        if (gi >= kGvStages && !mbar_wait(&empty[st], static_cast<uint32_t>(gi / kGvStages - 1) & 1u)) {
          report_error(err, kErrTimeoutProducer);
          *failed = 1;
          break;
        }
        fence_proxy_async_smem();
        // the group's rows are consecutive in W: one copy
        const int r0 = r_begin + gi * kGvRows;
        const uint32_t bytes = static_cast<uint32_t>(min(kGvRows, r_end - r0)) * kGvIn * 2;
        mbar_arrive_expect_tx(&full[st], bytes);
        bulk_load(ring + st * kGvStageBytes, W + static_cast<size_t>(r0) * kGvIn, bytes, &full[st]);
      }
      // the last stages' copies must land before the CTA exits
      for (int g2 = gi > kGvStages ? gi - kGvStages : 0; g2 < gi; ++g2)
        if (!mbar_wait(&full[g2 % kGvStages], static_cast<uint32_t>(g2 / kGvStages) & 1u)) {
          report_error(err, kErrTimeoutDrain);
          break;
        }
    }
  } else {
    // ---------------- consumers
    grid_dep_wait();
    float xa[2][16];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4* src = reinterpret_cast<const float4*>(x + r * kGvIn + h * 2048 + 8 * tid);
        const float4 v0 = src[0], v1 = src[1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) xa[r][h * 8 + i] = silu_in ? silu(v[i]) : v[i];
      }
    // after the butterfly, lanes 4 k .. 4 k + 3 hold sum number
    // (bit 4 of the lane) * 4 + (bit 3) * 2 + (bit 2) = row * 2 + x-row
    const int my_sum = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
    for (int gi = 0; gi < ngroups; ++gi) {
      const int st = gi % kGvStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], static_cast<uint32_t>(gi / kGvStages) & 1u))) {
        if (lane == 0) {
          report_error(err, kErrTimeoutEpilogue);
          *failed = 1;
        }
        break;
      }
      const int n = min(kGvRows, nrows - gi * kGvRows);
      const uint4* wst = reinterpret_cast<const uint4*>(ring + st * kGvStageBytes);
      float v[2 * kGvRows];
#pragma unroll
      for (int i = 0; i < kGvRows; ++i) {
        float a0 = 0.f, a1 = 0.f;
        if (i < n) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 w = wst[i * (kGvIn / 8) + h * 256 + tid];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float lo = __uint_as_float(ws[q] << 16);
              const float hi = __uint_as_float(ws[q] & 0xFFFF0000u);
              a0 = fmaf(hi, xa[0][h * 8 + 2 * q + 1], fmaf(lo, xa[0][h * 8 + 2 * q], a0));
              a1 = fmaf(hi, xa[1][h * 8 + 2 * q + 1], fmaf(lo, xa[1][h * 8 + 2 * q], a1));
            }
          }
        }
        v[2 * i] = a0;
        v[2 * i + 1] = a1;
      }
      // the stage is in registers: release it
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      // butterfly: at distance 16 each lane keeps half of the 8 sums (adding its
      // partner's copy of them) and hands over the other half; then 8 and 4; then a
      // plain sum over distances 2 and 1
      float w4[4], w2[2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool up = (lane & 16) != 0;
        const float give = up ? v[i] : v[i + 4];
        const float keep = up ? v[i + 4] : v[i];
        w4[i] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bool up = (lane & 8) != 0;
        const float give = up ? w4[i] : w4[i + 2];
        const float keep = up ? w4[i + 2] : w4[i];
        w2[i] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
      }
      float w1;
      {
        const bool up = (lane & 4) != 0;
        const float give = up ? w2[0] : w2[1];
        const float keep = up ? w2[1] : w2[0];
        w1 = keep + __shfl_xor_sync(0xffffffffu, give, 4);
      }
      w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
      w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
      if ((lane & 3) == 0 && (my_sum >> 1) < n)
        part[(warp * kGvMaxRows + gi * kGvRows + (my_sum >> 1)) * 2 + (my_sum & 1)] = w1;
    }
  }
  __syncthreads();
  if (*failed) return;
  grid_dep_wait();
  // every output of the CTA: its 8 warp sums in warp order, plus the bias
  for (int k = tid; k < 2 * nrows; k += kGvThreads) {
    const int row = k >> 1, r = k & 1;
    float sum = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kGvWarps; ++w2) sum += part[(w2 * kGvMaxRows + row) * 2 + r];
    const int o = r_begin + row;
    y[r * out_dim + o] = sum + bf16_bits_to_float(b[o]);
  }
}

// ---------------------------------------------------------------- norms

__device__ __forceinline__ float block_sum_256(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += red[i];
  __syncthreads();
  return s;
}

// ZeroCenterRMSNorm of text features: out = fp16(x / rms(x) * (1 + w)).
__global__ void __launch_bounds__(256) txt_prenorm_kernel(const float* __restrict__ txt,
                                                          const uint16_t* __restrict__ w,
                                                          act_t* __restrict__ out) {
  __shared__ float red[8];
  const int row = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(txt + static_cast<size_t>(row) * kHidden);
  float4 v[4];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = xr[threadIdx.x + 256 * i];
    ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  }
  const float rinv = rsqrtf(block_sum_256(ss, red) * (1.f / kHidden) + kEps);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = 4 * (threadIdx.x + 256 * i);
    const uint2 wb = *reinterpret_cast<const uint2*>(w + c);
    const float g0 = 1.f + __uint_as_float(wb.x << 16), g1 = 1.f + __uint_as_float(wb.x & 0xFFFF0000u);
    const float g2 = 1.f + __uint_as_float(wb.y << 16), g3 = 1.f + __uint_as_float(wb.y & 0xFFFF0000u);
    uint2 o;
    o.x = pack_f16x2(v[i].x * rinv * g0, v[i].y * rinv * g1);
    o.y = pack_f16x2(v[i].z * rinv * g2, v[i].w * rinv * g3);
    *reinterpret_cast<uint2*>(out + static_cast<size_t>(row) * kHidden + c) = o;
  }
}

// For a residual stream given directly: xa = fp16(x * (1 + s1[row])), plus the
// per-128-column sums of squares. One block per row; 16 consecutive columns per thread.
__global__ void __launch_bounds__(256) block_prep_kernel(const float* __restrict__ x, int n_text,
                                                         const float* __restrict__ mod,
                                                         act_t* __restrict__ xa, float* __restrict__ ssp) {
  const int row = blockIdx.x;
  const float* mrow = mod + (row < n_text ? kMod : 0);  // s1 is chunk 0
  const int c0 = threadIdx.x * 16;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(row) * kHidden + c0);
  const float4* sr = reinterpret_cast<const float4*>(mrow + c0);
  float ss = 0.f;
  uint32_t packed[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = xr[i];
    const float4 s = sr[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    packed[2 * i] = pack_f16x2(v.x * (1.f + s.x), v.y * (1.f + s.y));
    packed[2 * i + 1] = pack_f16x2(v.z * (1.f + s.z), v.w * (1.f + s.w));
  }
  uint4* dst = reinterpret_cast<uint4*>(xa + static_cast<size_t>(row) * kHidden + c0);
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  // 8 threads (16 columns each) cover one 128-column partial
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 7) == 0) ssp[static_cast<size_t>(row) * kSspParts + threadIdx.x / 8] = ss;
}

// ---------------------------------------------------------------- image projection

// x[r] = img[r] . W^T + b (64 -> 4096) for image rows (sampled-t modulation),
// xa = fp16(x * (1 + s1)), ssp = per-128-column sums of squares.
// Block: 256 columns (one per thread, its 64 weights in registers) x 64 rows.
constexpr int kImgRows = 64;
__global__ void __launch_bounds__(256) img_in_kernel(const float* __restrict__ img, int N,
                                                     const uint16_t* __restrict__ W, const uint16_t* __restrict__ b,
                                                     const float* __restrict__ mod, float* __restrict__ x,
                                                     act_t* __restrict__ xa, float* __restrict__ ssp) {
  __shared__ float rows[kImgRows][kPatch];
  __shared__ float red[kImgRows][8];
  const int col = blockIdx.x * 256 + threadIdx.x;
  const int r0 = blockIdx.y * kImgRows;
  const int nrows = min(kImgRows, N - r0);
  for (int i = threadIdx.x; i < kImgRows * kPatch; i += 256) {
    const int r = i / kPatch;
    rows[r][i % kPatch] = r < nrows ? img[static_cast<size_t>(r0 + r) * kPatch + i % kPatch] : 0.f;
  }
  float w[kPatch];
  const uint4* wr = reinterpret_cast<const uint4*>(W + static_cast<size_t>(col) * kPatch);
#pragma unroll
  for (int i = 0; i < kPatch / 8; ++i) {
    const uint4 v = wr[i];
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w[8 * i + 2 * j] = __uint_as_float(q[j] << 16);
      w[8 * i + 2 * j + 1] = __uint_as_float(q[j] & 0xFFFF0000u);
    }
  }
  const float bias = bf16_bits_to_float(b[col]);
  const float sc = 1.f + mod[col];  // image rows: sampled-t row, chunk s1
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 1
  for (int r = 0; r < nrows; ++r) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < kPatch; ++k) acc += rows[r][k] * w[k];
    acc += bias;
    const size_t idx = static_cast<size_t>(r0 + r) * kHidden + col;
    x[idx] = acc;
    xa[idx] = __float2half_rn(acc * sc);
    const float s = warp_sum(acc * acc);
    if (lane == 0) red[r][warp] = s;
  }
  __syncthreads();
  if (threadIdx.x < 2 * nrows) {
    // two partials per row: warps 0-3 cover this block's first 128 columns, 4-7 the rest
    const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) s += red[r][4 * half + i];
    ssp[static_cast<size_t>(r0 + r) * kSspParts + 2 * blockIdx.x + half] = s;
  }
}

// ---------------------------------------------------------------- output head

// vel[i] = (x[i] / rms(x[i])) . Wout^T + b, 4096 -> 64, with rms from the sum-of-squares
// partials. Block: 32 rows x 64 outputs, thread: 2 rows x 4 outputs (a float2 of x and a
// float4 of the k-major fp32 weight copy per k). K runs through shared memory 64 at a
// time; the next chunk is fetched into registers while the current one is multiplied.
// Each output sums its 4096 products in k order (one fma chain).
constexpr int kHeadRows = 32;
constexpr int kHeadK = 64;
constexpr int kHeadXPer = kHeadRows * kHeadK / 256;      // x values a thread stages per chunk (8)
constexpr int kHeadWPer = kHeadK * kPatch / 4 / 256;     // weight float4s a thread stages per chunk (4)
__global__ void __launch_bounds__(256) head_kernel(const float* __restrict__ x, int N, const float* __restrict__ ssp,
                                                   const float* __restrict__ wt, const uint16_t* __restrict__ b,
                                                   float* __restrict__ vel, int* err) {
  __shared__ __align__(16) float xs[kHeadK][kHeadRows + 2];  // [k][row], even stride: float2 reads
  __shared__ __align__(16) float ws[kHeadK][kPatch + 4];     // [k][output], float4 reads
  const int r0 = blockIdx.x * kHeadRows;
  const int tr = threadIdx.x >> 4;  // rows 2 tr, 2 tr + 1
  const int to = threadIdx.x & 15;  // outputs 4 to .. 4 to + 3
  float xr[kHeadXPer];
  float4 wr[kHeadWPer];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int i = 0; i < kHeadXPer; ++i) {
      const int e = threadIdx.x + 256 * i;
      const int r = e / kHeadK, k = e % kHeadK;
      xr[i] = (r0 + r) < N ? x[static_cast<size_t>(r0 + r) * kHidden + k0 + k] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kHeadWPer; ++i) {
      const int e = threadIdx.x + 256 * i;
      wr[i] = reinterpret_cast<const float4*>(wt + static_cast<size_t>(k0 + e / (kPatch / 4)) * kPatch)[e % (kPatch / 4)];
    }
  };
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  fetch(0);
#pragma unroll 1
  for (int k0 = 0; k0 < kHidden; k0 += kHeadK) {
#pragma unroll
    for (int i = 0; i < kHeadXPer; ++i) {
      const int e = threadIdx.x + 256 * i;
      xs[e % kHeadK][e / kHeadK] = xr[i];
    }
#pragma unroll
    for (int i = 0; i < kHeadWPer; ++i) {
      const int e = threadIdx.x + 256 * i;
      *reinterpret_cast<float4*>(&ws[e / (kPatch / 4)][4 * (e % (kPatch / 4))]) = wr[i];
    }
    __syncthreads();
    if (k0 + kHeadK < kHidden) fetch(k0 + kHeadK);
#pragma unroll 16
    for (int k = 0; k < kHeadK; ++k) {
      const float2 xv = *reinterpret_cast<const float2*>(&xs[k][2 * tr]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[k][4 * to]);
      acc[0][0] = fmaf(xv.x, wv.x, acc[0][0]);
      acc[0][1] = fmaf(xv.x, wv.y, acc[0][1]);
      acc[0][2] = fmaf(xv.x, wv.z, acc[0][2]);
      acc[0][3] = fmaf(xv.x, wv.w, acc[0][3]);
      acc[1][0] = fmaf(xv.y, wv.x, acc[1][0]);
      acc[1][1] = fmaf(xv.y, wv.y, acc[1][1]);
      acc[1][2] = fmaf(xv.y, wv.z, acc[1][2]);
      acc[1][3] = fmaf(xv.y, wv.w, acc[1][3]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = r0 + 2 * tr + rr;
    if (row >= N) continue;
    const float4* p = reinterpret_cast<const float4*>(ssp + static_cast<size_t>(row) * kSspParts);
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < kSspParts / 4; ++q) {
      const float4 v = p[q];
      s += v.x;
      s += v.y;
      s += v.z;
      s += v.w;
    }
    const float rinv = rsqrtf(s * (1.f / kHidden) + kEps);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v = acc[rr][j] * rinv + bf16_bits_to_float(b[4 * to + j]);
      vel[static_cast<size_t>(row) * kPatch + 4 * to + j] = v;  // the caller's buffer: 4-byte aligned only
      // guard: a non-finite velocity (e.g. an fp16 operand that left its range) is reported
      if (!isfinite(v)) report_error(err, kErrNonFinite);
    }
  }
}

// The output head's weight [64][4096] bf16 as a k-major fp32 copy [4096][64] (once at load).
__global__ void head_wt_kernel(const uint16_t* __restrict__ W, float* __restrict__ wt) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < kHidden * kPatch) wt[i] = bf16_bits_to_float(W[static_cast<size_t>(i % kPatch) * kHidden + i / kPatch]);
}

// ---------------------------------------------------------------- RoPE tables

// Value of axis table `axis` (width d = 16, 56, 56) at position pos, column k:
// omega = fl32(theta^(-2k/d)) in double; angle = fl32(fl32(pos) * omega);
// cos/sin evaluated in double and rounded once.
__device__ __forceinline__ void rope_value(int axis, int k, int pos, double theta, float& c, float& s) {
  const int d = axis == 0 ? 16 : 56;
  const float w = static_cast<float>(pow(theta, -(2.0 * k) / d));
  const float ang = __fmul_rn(static_cast<float>(pos), w);
  c = static_cast<float>(cos(static_cast<double>(ang)));
  s = static_cast<float>(sin(static_cast<double>(ang)));
}

__global__ void rope_axis_kernel(double theta, float* c0, float* s0, float* c1, float* s1, float* c2, float* s2) {
  const int row = blockIdx.x;   // 0..9215
  const int j = threadIdx.x;    // 0..63 -> axis columns 8 | 28 | 28
  const int pos = row - 1024;
  int axis, k, width;
  float *cp, *sp;
  if (j < 8) {
    axis = 0; k = j; width = 8; cp = c0; sp = s0;
  } else if (j < 36) {
    axis = 1; k = j - 8; width = 28; cp = c1; sp = s1;
  } else {
    axis = 2; k = j - 36; width = 28; cp = c2; sp = s2;
  }
  float c, s;
  rope_value(axis, k, pos, theta, c, s);
  if (cp) cp[static_cast<size_t>(row) * width + k] = c;
  if (sp) sp[static_cast<size_t>(row) * width + k] = s;
}

// Per-token rows: tokens [0, L) are text (i, i, i), [L, L + h*w) image.
__global__ void rope_tokens_kernel(int L, int h, int w, double theta, float* tc, float* ts, float* ic, float* is) {
  const int tok = blockIdx.x;
  const int j = threadIdx.x;  // 0..63
  int p0, p1, p2;
  if (tok < L) {
    p0 = p1 = p2 = tok;
  } else {
    const int n = tok - L;
    const int y = n / w, xx = n % w;
    p0 = L;
    p1 = y - (h - h / 2);
    p2 = xx - (w - w / 2);
  }
  int axis, k, pos;
  if (j < 8) {
    axis = 0; k = j; pos = p0;
  } else if (j < 36) {
    axis = 1; k = j - 8; pos = p1;
  } else {
    axis = 2; k = j - 36; pos = p2;
  }
  float c, s;
  rope_value(axis, k, pos, theta, c, s);
  float* cdst = tok < L ? tc : ic;
  float* sdst = tok < L ? ts : is;
  const size_t r = static_cast<size_t>(tok < L ? tok : tok - L);
  if (cdst) cdst[r * kRopeCols + j] = c;
  if (sdst) sdst[r * kRopeCols + j] = s;
}

// ---------------------------------------------------------------- sampler pieces

__global__ void euler_kernel(float* __restrict__ x, const float* __restrict__ vel, long long n, float s_i,
                             float s_next) {
  const float dt = __fsub_rn(s_next, s_i);
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i + 3 < n) {
    float4 a = *reinterpret_cast<float4*>(x + i);
    const float4 v = *reinterpret_cast<const float4*>(vel + i);
    a.x = __fadd_rn(a.x, __fmul_rn(dt, v.x));
    a.y = __fadd_rn(a.y, __fmul_rn(dt, v.y));
    a.z = __fadd_rn(a.z, __fmul_rn(dt, v.z));
    a.w = __fadd_rn(a.w, __fmul_rn(dt, v.w));
    *reinterpret_cast<float4*>(x + i) = a;
  } else {
    for (long long j = i; j < n; ++j) x[j] = __fadd_rn(x[j], __fmul_rn(dt, vel[j]));
  }
}

__global__ void cfg_combine_kernel(const float* __restrict__ pos, const float* __restrict__ neg, float g,
                                   float* __restrict__ out, long long n) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = __fadd_rn(neg[i], __fmul_rn(g, __fsub_rn(pos[i], neg[i])));
}

// DPM++ 2M step (float32, no contraction): D = x - sigma_i v; order 2 blends D with
// the previous step's D; order 0 returns D. D is kept for the next step.
__device__ __forceinline__ float dpm_one(float x, float v, float& dp, float sigma_i, int order, float a, float b,
                                         float c0, float c1) {
  const float D = __fsub_rn(x, __fmul_rn(sigma_i, v));
  float Dm = D;
  if (order == 2) Dm = __fsub_rn(__fmul_rn(c0, D), __fmul_rn(c1, dp));
  dp = D;
  return order == 0 ? D : __fadd_rn(__fmul_rn(a, x), __fmul_rn(b, Dm));
}

__global__ void dpmpp2m_kernel(float* __restrict__ x, const float* __restrict__ vel, float* __restrict__ dprev,
                               long long n, float sigma_i, int order, float a, float b, float c0, float c1) {
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i + 3 < n) {
    float4 xv = *reinterpret_cast<float4*>(x + i);
    const float4 v = *reinterpret_cast<const float4*>(vel + i);
    float4 dp = order == 2 ? *reinterpret_cast<const float4*>(dprev + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    xv.x = dpm_one(xv.x, v.x, dp.x, sigma_i, order, a, b, c0, c1);
    xv.y = dpm_one(xv.y, v.y, dp.y, sigma_i, order, a, b, c0, c1);
    xv.z = dpm_one(xv.z, v.z, dp.z, sigma_i, order, a, b, c0, c1);
    xv.w = dpm_one(xv.w, v.w, dp.w, sigma_i, order, a, b, c0, c1);
    *reinterpret_cast<float4*>(x + i) = xv;
    *reinterpret_cast<float4*>(dprev + i) = dp;
  } else {
    for (long long j = i; j < n; ++j) {
      float dp = order == 2 ? dprev[j] : 0.f;
      x[j] = dpm_one(x[j], vel[j], dp, sigma_i, order, a, b, c0, c1);
      dprev[j] = dp;
    }
  }
}

// ---------------------------------------------------------------- MXFP8 quantisation

// One thread per block of 32 values along K: the shared exponent
// e = floor(log2 max|v|) - 8 (8 = exponent of E4M3's largest normal, 448),
// clamped to [-127, 127], -127 for an all-zero block; each value becomes
// E4M3(v * 2^-e), rounded to nearest even and clamped to +-448. Scale byte e + 127
// goes to chunk (K-group k / 128, row group r / 128), byte
// (r % 32) * 16 + ((r % 128) / 32) * 4 + (k / 32) % 4.
template <bool BF16>
__global__ void quant_mx_kernel(const uint16_t* __restrict__ in, int rows, int K, int groups,
                                uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const int per_row = K / 32;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(rows) * per_row) return;
  const int r = static_cast<int>(idx / per_row);
  const int kb = static_cast<int>(idx - static_cast<long long>(r) * per_row);
  const uint4* src = reinterpret_cast<const uint4*>(in + static_cast<size_t>(r) * K + kb * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 w = src[i];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (BF16) {
        v[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
        v[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
      } else {
        const __half2 h = *reinterpret_cast<const __half2*>(&u[j]);
        const float2 f = __half22float2(h);
        v[8 * i + 2 * j] = f.x;
        v[8 * i + 2 * j + 1] = f.y;
      }
    }
  }
  sf[mx_sf_offset(r, kb, groups)] = mx_quant32(v, q + static_cast<size_t>(r) * K + kb * 32);
}

// ---------------------------------------------------------------- first-block cache

// r0 = x1 - x0 (block 0's residual), copies x1, and (when ref != nullptr) per-CTA sums
// of |r0 - ref| and |ref|: float within a thread, double across the CTA.
constexpr int kFbcThreads = 256;
__global__ void __launch_bounds__(kFbcThreads) fbc_residual_kernel(const float* __restrict__ x1,
                                                                   const float* __restrict__ x0,
                                                                   const float* __restrict__ ref,
                                                                   float* __restrict__ r0, float* __restrict__ x1c,
                                                                   long long n4, double2* __restrict__ partial) {
  float num = 0.f, den = 0.f;
  const long long stride = static_cast<long long>(gridDim.x) * kFbcThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kFbcThreads + threadIdx.x; i < n4; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(x1)[i];
    const float4 b = reinterpret_cast<const float4*>(x0)[i];
    const float4 r = make_float4(__fsub_rn(a.x, b.x), __fsub_rn(a.y, b.y), __fsub_rn(a.z, b.z), __fsub_rn(a.w, b.w));
    reinterpret_cast<float4*>(r0)[i] = r;
    reinterpret_cast<float4*>(x1c)[i] = a;
    if (ref) {
      const float4 p = reinterpret_cast<const float4*>(ref)[i];
      num += fabsf(r.x - p.x) + fabsf(r.y - p.y) + fabsf(r.z - p.z) + fabsf(r.w - p.w);
      den += fabsf(p.x) + fabsf(p.y) + fabsf(p.z) + fabsf(p.w);
    }
  }
  if (!ref) return;
  __shared__ double sn[kFbcThreads], sd[kFbcThreads];
  sn[threadIdx.x] = num;
  sd[threadIdx.x] = den;
  __syncthreads();
  for (int o = kFbcThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      sn[threadIdx.x] += sn[threadIdx.x + o];
      sd[threadIdx.x] += sd[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) partial[blockIdx.x] = make_double2(sn[0], sd[0]);
}

// Sums the per-CTA partials in a fixed order: out = {sum |r0 - ref|, sum |ref|}.
__global__ void __launch_bounds__(kFbcThreads) fbc_finish_kernel(const double2* __restrict__ partial, int n,
                                                                 double* __restrict__ out) {
  __shared__ double sn[kFbcThreads], sd[kFbcThreads];
  double a = 0.0, b = 0.0;
  for (int i = threadIdx.x; i < n; i += kFbcThreads) {
    a += partial[i].x;
    b += partial[i].y;
  }
  sn[threadIdx.x] = a;
  sd[threadIdx.x] = b;
  __syncthreads();
  for (int o = kFbcThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      sn[threadIdx.x] += sn[threadIdx.x + o];
      sd[threadIdx.x] += sd[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    out[0] = sn[0];
    out[1] = sd[0];
  }
}

// Skipped pass: x = x1 + rest per row, with the row's per-128-column sums of squares
// for the output head's norm. One CTA per row, 16 columns per thread.
__global__ void __launch_bounds__(256) fbc_apply_kernel(float* __restrict__ x, const float* __restrict__ rest,
                                                        float* __restrict__ ssp) {
  const size_t row = blockIdx.x;
  const int c0 = threadIdx.x * 16;
  float4* xr = reinterpret_cast<float4*>(x + row * kHidden + c0);
  const float4* rr = reinterpret_cast<const float4*>(rest + row * kHidden + c0);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = xr[i];
    const float4 r = rr[i];
    v.x = __fadd_rn(v.x, r.x);
    v.y = __fadd_rn(v.y, r.y);
    v.z = __fadd_rn(v.z, r.z);
    v.w = __fadd_rn(v.w, r.w);
    xr[i] = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 7) == 0) ssp[row * kSspParts + threadIdx.x / 8] = ss;
}

// Full pass: rest = x_last - x1 (the residual of blocks 1..last).
__global__ void fbc_rest_kernel(const float* __restrict__ xl, const float* __restrict__ x1c, float* __restrict__ rest,
                                long long n4) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(xl)[i];
    const float4 b = reinterpret_cast<const float4*>(x1c)[i];
    reinterpret_cast<float4*>(rest)[i] =
        make_float4(__fsub_rn(a.x, b.x), __fsub_rn(a.y, b.y), __fsub_rn(a.z, b.z), __fsub_rn(a.w, b.w));
  }
}

// x[t, c] = z[c, t] for t < h*w, c < 64 (32x32 tiles through shared memory).
__global__ void pack_noise_kernel(const float* __restrict__ z, int T, float* __restrict__ x) {
  __shared__ float tile[32][33];
  const int t0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i, t = t0 + threadIdx.x;
    tile[i][threadIdx.x] = t < T ? z[static_cast<size_t>(c) * T + t] : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int t = t0 + i, c = c0 + threadIdx.x;
    if (t < T) x[static_cast<size_t>(t) * kPatch + c] = tile[threadIdx.x][i];
  }
}

// In place bf16 -> fp16 conversion of a weight tensor, two values per thread
// step. fp16 holds every bf16 value of magnitude 2^-14..65504 exactly; smaller
// ones round to fp16 subnormals (error < 2^-25); larger ones are counted.
__global__ void bf16_to_f16_kernel(uint32_t* w, size_t pairs, unsigned int* overflow) {
  unsigned int bad = 0;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < pairs;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint32_t v = w[i];
    const float lo = __uint_as_float(v << 16);
    const float hi = __uint_as_float(v & 0xFFFF0000u);
    bad += (fabsf(lo) > 65504.f) + (fabsf(hi) > 65504.f);
    w[i] = pack_f16x2(lo, hi);
  }
  if (bad) atomicAdd(overflow, bad);
}

// Largest magnitude of an fp16 tensor (n a multiple of 8, 16-byte aligned) into
// *out with an atomic max on the float's bits (non-negative floats order like
// their bit patterns); a NaN counts as +inf, so an overflow cannot hide.
__global__ void absmax_f16_kernel(const uint4* a, long long n8, float* out) {
  float m = 0.f;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 w = a[i];
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 hv = *reinterpret_cast<const __half2*>(&v[k]);
      const float2 f = __half22float2(hv);
      const float a0 = fabsf(f.x), a1 = fabsf(f.y);
      m = fmaxf(m, a0 != a0 ? INFINITY : a0);
      m = fmaxf(m, a1 != a1 ? INFINITY : a1);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<int*>(out), __float_as_int(m));
}

}  // namespace

// ---------------------------------------------------------------- launchers

cudaError_t launch_timestep_embed(float t, float* e, cudaStream_t s) {
  timestep_embed_kernel<<<1, 128, 0, s>>>(t, e);
  return cudaGetLastError();
}

cudaError_t launch_gemv2(const float* x, int in_dim, const uint16_t* W, const uint16_t* b, int out_dim, float* y,
                         int silu_in, int* err, bool weights_preloaded, cudaStream_t s) {
  if (out_dim <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (in_dim == kGvIn) {
    // bulk copies and vector loads need 16-byte aligned W and x
    if ((reinterpret_cast<uintptr_t>(W) & 15) != 0 || (reinterpret_cast<uintptr_t>(x) & 15) != 0)
      return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr_done{0};
    e = ensure_smem_limit(gemv_stream_kernel, kGvSmem, attr_done);
    if (e != cudaSuccess) return e;
    // one CTA per SM, or more so that no CTA has more than kGvMaxRows rows
    int grid = out_dim < sms ? out_dim : sms;
    const int need = (out_dim + kGvMaxRows - 1) / kGvMaxRows;
    if (grid < need) grid = need;
    if (weights_preloaded)
      return launch_dependent(gemv_stream_kernel, dim3(grid), dim3(kGvThreads), kGvSmem, s, x, W, b, out_dim, y,
                              silu_in, err);
    gemv_stream_kernel<<<grid, kGvThreads, kGvSmem, s>>>(x, W, b, out_dim, y, silu_in, err);
    return cudaGetLastError();
  }
  const size_t smem = 2 * static_cast<size_t>(in_dim) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gemv2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  // four blocks of 8 warps per SM (or fewer if there are fewer output groups)
  const int groups = (out_dim + kOutPerWarp - 1) / kOutPerWarp;
  const int grid = groups < 4 * sms ? groups : 4 * sms;
  gemv2_kernel<<<grid, 256, smem, s>>>(x, in_dim, W, b, out_dim, y, silu_in);
  return cudaGetLastError();
}

cudaError_t launch_txt_prenorm(const float* txt, int L, const uint16_t* w, act_t* out, cudaStream_t s) {
  if (L <= 0) return cudaSuccess;
  txt_prenorm_kernel<<<L, 256, 0, s>>>(txt, w, out);
  return cudaGetLastError();
}

cudaError_t launch_block_prep(const float* x, int R, int n_text, const float* mod, act_t* xa, float* ssp,
                              cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  block_prep_kernel<<<R, 256, 0, s>>>(x, n_text, mod, xa, ssp);
  return cudaGetLastError();
}

cudaError_t launch_img_in(const float* img, int N, const uint16_t* W, const uint16_t* b, const float* mod, float* x,
                          act_t* xa, float* ssp, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  dim3 grid(kHidden / 256, (N + kImgRows - 1) / kImgRows);
  img_in_kernel<<<grid, 256, 0, s>>>(img, N, W, b, mod, x, xa, ssp);
  return cudaGetLastError();
}

cudaError_t launch_head(const float* x, int N, const float* ssp, const float* wt, const uint16_t* b, float* vel,
                        int* err, cudaStream_t s) {
  if (N <= 0) return cudaSuccess;
  head_kernel<<<(N + kHeadRows - 1) / kHeadRows, 256, 0, s>>>(x, N, ssp, wt, b, vel, err);
  return cudaGetLastError();
}

cudaError_t launch_head_wt(const uint16_t* W, float* wt, cudaStream_t s) {
  head_wt_kernel<<<(kHidden * kPatch + 255) / 256, 256, 0, s>>>(W, wt);
  return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16(uint16_t* w, size_t n, unsigned int* overflow, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const size_t pairs = n / 2;  // weight tensors here have an even element count
  const size_t want = (pairs + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 148 * 32 ? want : 148 * 32);
  bf16_to_f16_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<uint32_t*>(w), pairs, overflow);
  return cudaGetLastError();
}

cudaError_t launch_absmax_f16(const act_t* a, long long n, float* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long long n8 = n / 8;
  const long long want = (n8 + 255) / 256;
  absmax_f16_kernel<<<static_cast<unsigned>(want < 1216 ? want : 1216), 256, 0, s>>>(reinterpret_cast<const uint4*>(a),
                                                                                      n8, out);
  return cudaGetLastError();
}

cudaError_t launch_euler(float* x, const float* vel, long long n, float s_i, float s_next, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long long threads = (n + 3) / 4;
  euler_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(x, vel, n, s_i, s_next);
  return cudaGetLastError();
}

cudaError_t launch_dpmpp2m(float* x, const float* vel, float* dprev, long long n, float sigma_i, int order, float a,
                           float b, float c0, float c1, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const long long threads = (n + 3) / 4;
  dpmpp2m_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(x, vel, dprev, n, sigma_i, order, a, b,
                                                                             c0, c1);
  return cudaGetLastError();
}

cudaError_t launch_quant_mx(const uint16_t* in, bool bf16, int rows, int K, uint8_t* q, uint8_t* sf,
                            cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (K % 128 != 0) return cudaErrorInvalidValue;
  const long long n = static_cast<long long>(rows) * (K / 32);
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  const int groups = (rows + 127) / 128;
  if (bf16)
    quant_mx_kernel<true><<<blocks, 256, 0, s>>>(in, rows, K, groups, q, sf);
  else
    quant_mx_kernel<false><<<blocks, 256, 0, s>>>(in, rows, K, groups, q, sf);
  return cudaGetLastError();
}

cudaError_t launch_fbc_residual(const float* x1, const float* x0, const float* ref, float* r0, float* x1c, int rows,
                                int grid, double2* partial, double* out, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const long long n4 = static_cast<long long>(rows) * kHidden / 4;
  fbc_residual_kernel<<<grid, kFbcThreads, 0, s>>>(x1, x0, ref, r0, x1c, n4, partial);
  if (ref) fbc_finish_kernel<<<1, kFbcThreads, 0, s>>>(partial, grid, out);
  return cudaGetLastError();
}

cudaError_t launch_fbc_apply(float* x, const float* rest, float* ssp, int rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  fbc_apply_kernel<<<rows, 256, 0, s>>>(x, rest, ssp);
  return cudaGetLastError();
}

cudaError_t launch_fbc_rest(const float* xl, const float* x1c, float* rest, int rows, int grid, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  fbc_rest_kernel<<<grid, 256, 0, s>>>(xl, x1c, rest, static_cast<long long>(rows) * kHidden / 4);
  return cudaGetLastError();
}

cudaError_t launch_rope_axis(float theta, float* c0, float* s0, float* c1, float* s1, float* c2, float* s2,
                             cudaStream_t s) {
  rope_axis_kernel<<<9216, 64, 0, s>>>(static_cast<double>(theta), c0, s0, c1, s1, c2, s2);
  return cudaGetLastError();
}

cudaError_t launch_rope_tokens(int L, int h, int w, float theta, float* tc, float* ts, float* ic, float* is,
                               cudaStream_t s) {
  const int T = L + h * w;
  if (T <= 0) return cudaSuccess;
  rope_tokens_kernel<<<T, 64, 0, s>>>(L, h, w, static_cast<double>(theta), tc, ts, ic, is);
  return cudaGetLastError();
}

cudaError_t launch_cfg_combine(const float* pos, const float* neg, float g, float* out, long long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  cfg_combine_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(pos, neg, g, out, n);
  return cudaGetLastError();
}

cudaError_t launch_pack_noise(const float* z, int h, int w, float* x, cudaStream_t s) {
  const int T = h * w;
  if (T <= 0) return cudaSuccess;
  dim3 grid((T + 31) / 32, kPatch / 32);
  pack_noise_kernel<<<grid, dim3(32, 8), 0, s>>>(z, T, x);
  return cudaGetLastError();
}

}  // namespace qi
