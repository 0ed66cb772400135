// Hybrid training backward with the L1 term ("Sparser, Faster, Lighter
// Transformer Language Models", section 2.B.3: custom sparse-to-dense and
// dense-to-sparse matmuls in the backward pass over the hybrid format; the
// L1 penalty with coefficient 2e-5 on the FFN activations comes from the
// news article "Sakana AI and NVIDIA TwELL boosts LLM training speed by
// 21.9%", recipe list).
//
// With a = h * u and the loss L(y) + lambda * sum(h):
//   da = dy W_d^T, du = da h, dz = da u + lambda (active entries only),
//   dx = dz W_g^T + du W_u^T, dW_g = x^T dz, dW_u = x^T du, dW_d = a^T dy.
//
// ELL rows (CUDA cores):
//   count     one warp per ELL row: per-neuron entry counts (atomics)
//   scan      one CTA: per-neuron offsets (CSC), cursors = offsets
//   ell_bwd   one warp per ELL row: neuron rows W_d[j], W_g^T[j], W_u^T[j]
//             staged by cp.async.bulk; da = dy_t . W_d[j, :] (dense-to-
//             sparse), dx_t += dz W_g^T[j] + du W_u^T[j] (sparse-to-dense);
//             one record (t, dz, du, a) per entry is appended to neuron j's
//             CSC segment
//   dw        one CTA per neuron j: walks its records and accumulates the
//             sparse-to-dense products dW_g^T[j] = sum dz x_t,
//             dW_u^T[j] = sum du x_t, dW_d[j] = sum a dy_t (stored)
// Dense overflow rows (tensor cores, fp32 operands split into bf16 hi+lo):
//   G3  dA = dY_ov W_d^T, epilogue dz, du (split)          -> G
//   G4  dx[dense rows] = dz W_g^T + du W_u^T                (W_g, W_u staged
//       transposed; K split in ranges of <= 4096 summed with fp32 atomics)
//   G5-G7  dW_g^T += dz^T X_ov, dW_u^T += du^T X_ov, dW_d += a^T dY_ov
//       (operands staged transposed, K = number of dense rows, read on the
//       device)
// dW rows are written by `dw` first and accumulated into by G5-G7; dx rows
// of ELL and dense tokens are written by ell_bwd and G4 respectively.
#include "bounds.cuh"
#include "gemm.cuh"
#include "hybrid.cuh"
#include "ptx.cuh"

namespace twell {
namespace {

constexpr int kWarps = 8;
constexpr int kListCap = 64;
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 231168;  // within the 227 KB opt-in limit

struct BwdParams {
  const uint16_t* x;
  const float* dy;
  const uint16_t* Wg_t;
  const uint16_t* Wu_t;
  const uint16_t* Wd;
  const float* u_ell;
  const float* ell_val;
  const uint8_t* ell_col;
  const uint8_t* ell_cnt;
  const int32_t* ell_rows;
  const int32_t* n_ell;
  int32_t T, D, F, n_t, C;
  float lambda;
  float* dx;
  float* dWg_t;
  float* dWu_t;
  float* dWd;
  int32_t* cnt;
  int32_t* offs;
  int32_t* cursor;
  BwdRecord* rec;
  int32_t stages;
  int32_t warp_bytes;
  int32_t* status;
};

struct BEntry {
  int32_t j;
  float h;
  int32_t pos;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 pairs in a 64-bit register pair, for the packed pair FMA (sm_100+)
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d = a * b + d on fp32 pairs
__device__ __forceinline__ void fma2(f32x2& d, f32x2 a, f32x2 b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

__device__ __forceinline__ f32x2 widen(uint32_t w) { return pack2(bf16lo(w), bf16hi(w)); }

__global__ void __launch_bounds__(256) count_kernel(const BwdParams p) {
  const int lane = threadIdx.x & 31;
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (i >= *p.n_ell) return;
  const size_t rt0 = static_cast<size_t>(i) * p.n_t;
  for (int k = lane; k < p.n_t; k += 32) {
    int c = p.ell_cnt[rt0 + k];
    if (!in_bounds(c, p.C + 1, p.status)) c = 0;
    const uint8_t* col = p.ell_col + (rt0 + k) * p.C;
    for (int s = 0; s < c; ++s) {
      const int j = k * TWELL_TILE + col[s];
      if (in_bounds(j, p.F, p.status)) atomicAdd(&p.cnt[j], 1);
    }
  }
}

__global__ void __launch_bounds__(1024) offsets_kernel(const BwdParams p) {
  __shared__ int32_t part[1024];
  const int tid = threadIdx.x;
  const int per = (p.F + 1023) / 1024;
  const int j0 = tid * per;
  const int j1 = min(p.F, j0 + per);
  int sum = 0;
  for (int j = j0; j < j1; ++j) sum += p.cnt[j];
  part[tid] = sum;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    const int v = tid >= d ? part[tid - d] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = part[tid] - sum;
  for (int j = j0; j < j1; ++j) {
    p.offs[j] = run;
    p.cursor[j] = run;
    run += p.cnt[j];
  }
  if (tid == 1023) p.offs[p.F] = part[1023];
}

template <int NC, bool EXACT>
__global__ void __launch_bounds__(kWarps * 32, 1) ell_bwd_kernel(const BwdParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int P = p.stages;
  const int D = p.D;
  const int nch = D >> 3;
  const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;
  const uint32_t stage_bytes = 3u * row_bytes;

  uint8_t* wbase = smem + static_cast<size_t>(wid) * p.warp_bytes;
  uint8_t* stages = wbase;  // P x [W_d row | W_g^T row | W_u^T row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + static_cast<size_t>(P) * stage_bytes);
  BEntry* list = reinterpret_cast<BEntry*>(bars + kMaxStages);

  if (lane == 0) {
    for (int s = 0; s < P; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  auto own = [&](int i) { return EXACT || (lane + 32 * i) < nch; };
  uint32_t seq = 0;
  auto issue = [&](const BEntry& e, uint32_t n) {
    const int s = static_cast<int>(n % static_cast<uint32_t>(P));
    uint8_t* dst = stages + static_cast<size_t>(s) * stage_bytes;
    const size_t off = static_cast<size_t>(clamp_index(e.j, p.F, p.status)) * D;
    ptx::mbar_arrive_expect_tx(&bars[s], stage_bytes);
    ptx::bulk_load(dst, p.Wd + off, row_bytes, &bars[s]);
    ptx::bulk_load(dst + row_bytes, p.Wg_t + off, row_bytes, &bars[s]);
    ptx::bulk_load(dst + 2 * row_bytes, p.Wu_t + off, row_bytes, &bars[s]);
  };

  // contiguous row range per CTA, handed to its warps in order of completion
  __shared__ int next_row;
  const int n_rows = *p.n_ell;
  const int i_begin = static_cast<int>(static_cast<long long>(n_rows) * blockIdx.x / gridDim.x);
  const int i_end =
      static_cast<int>(static_cast<long long>(n_rows) * (blockIdx.x + 1) / gridDim.x);
  if (threadIdx.x == 0) next_row = 0;
  __syncthreads();
  for (;;) {
    int take = 0;
    if (lane == 0) take = atomicAdd(&next_row, 1);
    const int i = i_begin + __shfl_sync(0xffffffffu, take, 0);
    if (i >= i_end) break;
    const int t = p.ell_rows[i];
    if (!in_bounds(t, p.T, p.status)) continue;  // warp-uniform
    f32x2 dyf[NC][4];  // dy_t, fp32 pairs
    f32x2 acc[NC][4];  // dx_t accumulator, fp32 pairs
    const float* dyr = p.dy + static_cast<size_t>(t) * D;
#pragma unroll
    for (int q = 0; q < NC; ++q) {
      if (own(q)) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(dyr + 8 * (lane + 32 * q)));
        const float4 b = __ldg(reinterpret_cast<const float4*>(dyr + 8 * (lane + 32 * q)) + 1);
        dyf[q][0] = pack2(a.x, a.y);
        dyf[q][1] = pack2(a.z, a.w);
        dyf[q][2] = pack2(b.x, b.y);
        dyf[q][3] = pack2(b.z, b.w);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) dyf[q][e] = 0ull;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[q][e] = 0ull;
    }

    const size_t rt0 = static_cast<size_t>(i) * p.n_t;
    for (int kb = 0; kb < p.n_t; kb += 32) {
      const int k = kb + lane;
      int n = k < p.n_t ? p.ell_cnt[rt0 + k] : 0;
      if (!in_bounds(n, p.C + 1, p.status)) n = 0;
      int off = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, off, d);
        if (lane >= d) off += v;
      }
      const int total = __shfl_sync(0xffffffffu, off, 31);
      off -= n;
      for (int base = 0; base < total; base += kListCap) {
        if (n > 0 && off + n > base && off < base + kListCap) {
          const size_t so = (rt0 + k) * static_cast<size_t>(p.C);
          const int s0 = max(0, base - off);
          const int s1 = min(n, base + kListCap - off);
          for (int s = s0; s < s1; ++s)
            list[off + s - base] = BEntry{k * TWELL_TILE + p.ell_col[so + s],
                                          p.ell_val[so + s], static_cast<int32_t>(so + s)};
        }
        __syncwarp();
        const int m = min(kListCap, total - base);
        if (lane == 0) {
          const int pre = min(P, m);
          for (int e = 0; e < pre; ++e) issue(list[e], seq + e);
        }
        for (int e = 0; e < m; ++e) {
          const uint32_t n_e = seq + e;
          const int s = static_cast<int>(n_e % static_cast<uint32_t>(P));
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars[s], (n_e / P) & 1u))) {
            // wait (bounded) for this warp's row copies still in flight
            // (entries e .. e + P - 1) before leaving
            if (lane == 0) {
              atomicOr(p.status, TWELL_FLAG_TIMEOUT);
              for (int r = e; r < min(m, e + P); ++r) {
                const uint32_t n_r = seq + r;
                if (!ptx::mbar_wait(&bars[n_r % static_cast<uint32_t>(P)], (n_r / P) & 1u)) break;
              }
            }
            __syncwarp();
            return;
          }
          const BEntry en = list[e];
          const uint4* sd = reinterpret_cast<const uint4*>(stages + static_cast<size_t>(s) *
                                                                        stage_bytes);
          const uint4* sg = sd + nch;
          const uint4* su = sg + nch;
          f32x2 pp[4] = {0ull, 0ull, 0ull, 0ull};  // eight independent partial sums
#pragma unroll
          for (int q = 0; q < NC; ++q) {
            if (own(q)) {
              const uint4 a = sd[lane + 32 * q];
              const uint32_t a4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
              for (int r = 0; r < 4; ++r) fma2(pp[r], dyf[q][r], widen(a4[r]));
            }
          }
          float p0, p1, p2, p3, p4, p5, p6, p7;
          unpack2(pp[0], p0, p1);
          unpack2(pp[1], p2, p3);
          unpack2(pp[2], p4, p5);
          unpack2(pp[3], p6, p7);
          float da = ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) da += __shfl_xor_sync(0xffffffffu, da, o);
          const float u =
              p.u_ell[clamp_index(en.pos, static_cast<long long>(p.T) * p.n_t * p.C, p.status)];
          const float du = da * en.h;
          const float dz = fmaf(da, u, p.lambda);
          const f32x2 dz2 = pack2(dz, dz);
          const f32x2 du2 = pack2(du, du);
#pragma unroll
          for (int q = 0; q < NC; ++q) {
            if (own(q)) {
              const uint4 g = sg[lane + 32 * q];
              const uint4 w = su[lane + 32 * q];
              const uint32_t g4[4] = {g.x, g.y, g.z, g.w};
              const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                fma2(acc[q][r], dz2, widen(g4[r]));
                fma2(acc[q][r], du2, widen(w4[r]));
              }
            }
          }
          if (lane == 0 && in_bounds(en.j, p.F, p.status)) {
            const int r = atomicAdd(&p.cursor[en.j], 1);
            if (in_bounds(r, static_cast<long long>(p.T) * p.n_t * p.C, p.status))
              p.rec[r] = BwdRecord{t, dz, du, en.h * u};
          }
          __syncwarp();
          if (lane == 0 && e + P < m) {
            ptx::fence_proxy_async_smem();
            issue(list[e + P], n_e + P);
          }
        }
        seq += static_cast<uint32_t>(m);
        __syncwarp();
      }
    }
    float* dxr = p.dx + static_cast<size_t>(t) * D;
#pragma unroll
    for (int q = 0; q < NC; ++q) {
      if (own(q)) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) unpack2(acc[q][e], v[2 * e], v[2 * e + 1]);
        float4* o = reinterpret_cast<float4*>(dxr + 8 * (lane + 32 * q));
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
      }
    }
  }
}

// One CTA per neuron j; thread c owns columns [8c, 8c+8).
__global__ void __launch_bounds__(384) dw_kernel(const BwdParams p) {
  const int j = blockIdx.x;
  const int c = threadIdx.x;
  const int D = p.D;
  const bool own = 8 * c < D;
  float g[8], w[8], d[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) g[e] = w[e] = d[e] = 0.0f;
  const long long n_rec = static_cast<long long>(p.T) * p.n_t * p.C;
  int r0 = p.offs[j];
  int r1 = p.offs[j + 1];
  if (!in_bounds(r0, n_rec + 1, p.status) || !in_bounds(r1, n_rec + 1, p.status) || r1 < r0)
    r0 = r1 = 0;
  if (own) {
    int r = r0;
    for (; r + 2 <= r1; r += 2) {
      BwdRecord a = p.rec[r];
      BwdRecord b = p.rec[r + 1];
      a.t = static_cast<int32_t>(clamp_index(a.t, p.T, p.status));
      b.t = static_cast<int32_t>(clamp_index(b.t, p.T, p.status));
      const uint4 xa = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(a.t) * D) + c);
      const uint4 xb = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(b.t) * D) + c);
      const float4* ya = reinterpret_cast<const float4*>(p.dy + static_cast<size_t>(a.t) * D) + 2 * c;
      const float4* yb = reinterpret_cast<const float4*>(p.dy + static_cast<size_t>(b.t) * D) + 2 * c;
      const float4 ya0 = __ldg(ya), ya1 = __ldg(ya + 1), yb0 = __ldg(yb), yb1 = __ldg(yb + 1);
      const uint32_t xa4[4] = {xa.x, xa.y, xa.z, xa.w};
      const uint32_t xb4[4] = {xb.x, xb.y, xb.z, xb.w};
      const float yav[8] = {ya0.x, ya0.y, ya0.z, ya0.w, ya1.x, ya1.y, ya1.z, ya1.w};
      const float ybv[8] = {yb0.x, yb0.y, yb0.z, yb0.w, yb1.x, yb1.y, yb1.z, yb1.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float xal = bf16lo(xa4[e]), xah = bf16hi(xa4[e]);
        const float xbl = bf16lo(xb4[e]), xbh = bf16hi(xb4[e]);
        g[2 * e] = fmaf(b.dz, xbl, fmaf(a.dz, xal, g[2 * e]));
        g[2 * e + 1] = fmaf(b.dz, xbh, fmaf(a.dz, xah, g[2 * e + 1]));
        w[2 * e] = fmaf(b.du, xbl, fmaf(a.du, xal, w[2 * e]));
        w[2 * e + 1] = fmaf(b.du, xbh, fmaf(a.du, xah, w[2 * e + 1]));
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) d[e] = fmaf(b.a, ybv[e], fmaf(a.a, yav[e], d[e]));
    }
    for (; r < r1; ++r) {
      BwdRecord a = p.rec[r];
      a.t = static_cast<int32_t>(clamp_index(a.t, p.T, p.status));
      const uint4 xa = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(a.t) * D) + c);
      const float4* ya = reinterpret_cast<const float4*>(p.dy + static_cast<size_t>(a.t) * D) + 2 * c;
      const float4 ya0 = __ldg(ya), ya1 = __ldg(ya + 1);
      const uint32_t xa4[4] = {xa.x, xa.y, xa.z, xa.w};
      const float yav[8] = {ya0.x, ya0.y, ya0.z, ya0.w, ya1.x, ya1.y, ya1.z, ya1.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        g[2 * e] = fmaf(a.dz, bf16lo(xa4[e]), g[2 * e]);
        g[2 * e + 1] = fmaf(a.dz, bf16hi(xa4[e]), g[2 * e + 1]);
        w[2 * e] = fmaf(a.du, bf16lo(xa4[e]), w[2 * e]);
        w[2 * e + 1] = fmaf(a.du, bf16hi(xa4[e]), w[2 * e + 1]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) d[e] = fmaf(a.a, yav[e], d[e]);
    }
    const size_t o = static_cast<size_t>(j) * D + 8 * c;
    float4* og = reinterpret_cast<float4*>(p.dWg_t + o);
    float4* ou = reinterpret_cast<float4*>(p.dWu_t + o);
    float4* od = reinterpret_cast<float4*>(p.dWd + o);
    og[0] = make_float4(g[0], g[1], g[2], g[3]);
    og[1] = make_float4(g[4], g[5], g[6], g[7]);
    ou[0] = make_float4(w[0], w[1], w[2], w[3]);
    ou[1] = make_float4(w[4], w[5], w[6], w[7]);
    od[0] = make_float4(d[0], d[1], d[2], d[3]);
    od[1] = make_float4(d[4], d[5], d[6], d[7]);
  }
}

template <int NC>
twell_status launch_ell_bwd(BwdParams p, const DeviceInfo& dev, cudaStream_t s) {
  const int stage_bytes = 6 * p.D;
  const int fixed = kMaxStages * 8 + kListCap * static_cast<int>(sizeof(BEntry));
  const int budget = kSmemBudget < dev.max_smem_optin ? kSmemBudget : dev.max_smem_optin;
  int P = (budget / kWarps - fixed) / stage_bytes;
  if (P > kMaxStages) P = kMaxStages;
  if (P < 1) return TWELL_ERR_UNSUPPORTED;
  p.stages = P;
  p.warp_bytes = (P * stage_bytes + fixed + 15) & ~15;
  const int smem = kWarps * p.warp_bytes;
  auto kern = p.D == 256 * NC ? ell_bwd_kernel<NC, true> : ell_bwd_kernel<NC, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return TWELL_ERR_CUDA;
  const long long want = (static_cast<long long>(p.T) + kWarps - 1) / kWarps;
  const int grid = static_cast<int>(want < dev.sm_count ? want : dev.sm_count);
  kern<<<grid, kWarps * 32, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

twell_status ell_bwd(const BwdParams& p, const DeviceInfo& dev, cudaStream_t s) {
#define TWELL_NC_CASE(n) \
  case n:                \
    return launch_ell_bwd<n>(p, dev, s);
  switch ((p.D + 255) / 256) {
    TWELL_NC_CASE(1)
    TWELL_NC_CASE(2)
    TWELL_NC_CASE(3)
    TWELL_NC_CASE(4)
    TWELL_NC_CASE(5)
    TWELL_NC_CASE(6)
    TWELL_NC_CASE(7)
    TWELL_NC_CASE(8)
    TWELL_NC_CASE(9)
    TWELL_NC_CASE(10)
    TWELL_NC_CASE(11)
    TWELL_NC_CASE(12)
    default:
      return TWELL_ERR_UNSUPPORTED;
  }
#undef TWELL_NC_CASE
}

}  // namespace
}  // namespace twell

extern "C" twell_status hybrid_ffn_bwd(const uint16_t* x, const hybrid_t* h, const float* u_ell,
                                       const float* U_dense, const uint16_t* Wg_t,
                                       const uint16_t* Wu_t, const uint16_t* Wd, int32_t D,
                                       const float* dy, float l1_coeff, float* dx, float* dWg_t,
                                       float* dWu_t, float* dWd, void* ws, size_t ws_bytes,
                                       int32_t* status_dev, void* stream) {
  using namespace twell;
  if (h == nullptr) return TWELL_ERR_INVALID;
  const int32_t T = h->T, F = h->F;
  if (T < 0 || F <= 0 || F % TWELL_TILE != 0 || D <= 0 || D % 8 != 0) return TWELL_ERR_INVALID;
  twell_status st = check_hybrid(h, T, F);
  if (st != TWELL_OK) return st;
  if (!Wg_t || !Wu_t || !Wd || !dWg_t || !dWu_t || !dWd || !status_dev) return TWELL_ERR_INVALID;
  if (!aligned16(Wg_t) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(dWg_t) ||
      !aligned16(dWu_t) || !aligned16(dWd))
    return TWELL_ERR_INVALID;
  if (D > 256 * 12) return TWELL_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(2, T, D, F, h->cap, h->max_dense);
  if (T > 0) {
    if (!x || !dy || !dx || !u_ell || !ws || ws_bytes < L.bytes) return TWELL_ERR_INVALID;
    if (h->max_dense > 0 && !U_dense) return TWELL_ERR_INVALID;
    if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(u_ell) ||
        (U_dense && !aligned16(U_dense)) || (reinterpret_cast<uintptr_t>(ws) & 255u))
      return TWELL_ERR_INVALID;
  }
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t wbytes = static_cast<size_t>(F) * D * sizeof(float);
  if (T == 0) {  // no tokens: every gradient is zero
    if (cudaMemsetAsync(dWg_t, 0, wbytes, s) != cudaSuccess ||
        cudaMemsetAsync(dWu_t, 0, wbytes, s) != cudaSuccess ||
        cudaMemsetAsync(dWd, 0, wbytes, s) != cudaSuccess)
      return TWELL_ERR_CUDA;
    return TWELL_OK;
  }

  uint8_t* w = static_cast<uint8_t*>(ws);
  BwdParams p{};
  p.x = x;
  p.dy = dy;
  p.Wg_t = Wg_t;
  p.Wu_t = Wu_t;
  p.Wd = Wd;
  p.u_ell = u_ell;
  p.ell_val = h->ell_val;
  p.ell_col = h->ell_col;
  p.ell_cnt = h->ell_cnt;
  p.ell_rows = h->ell_rows;
  p.n_ell = h->n_ell;
  p.T = T;
  p.D = D;
  p.F = F;
  p.n_t = F / TWELL_TILE;
  p.C = h->cap;
  p.lambda = l1_coeff;
  p.dx = dx;
  p.dWg_t = dWg_t;
  p.dWu_t = dWu_t;
  p.dWd = dWd;
  p.cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  p.offs = reinterpret_cast<int32_t*>(w + L.offs);
  p.cursor = reinterpret_cast<int32_t*>(w + L.cursor);
  p.rec = reinterpret_cast<BwdRecord*>(w + L.records);
  p.status = status_dev;

  // ---- ELL rows
  if (cudaMemsetAsync(p.cnt, 0, static_cast<size_t>(F) * sizeof(int32_t), s) != cudaSuccess)
    return TWELL_ERR_CUDA;
  const int warp_blocks = static_cast<int>((static_cast<long long>(T) * 32 + 255) / 256);
  count_kernel<<<warp_blocks, 256, 0, s>>>(p);
  offsets_kernel<<<1, 1024, 0, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  if ((st = ell_bwd(p, dev, s)) != TWELL_OK) return st;
  const int dw_threads = ((D / 8) + 31) / 32 * 32;
  dw_kernel<<<F, dw_threads, 0, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return TWELL_ERR_CUDA;
  if (h->max_dense == 0) return TWELL_OK;

  // ---- dense overflow rows
  return dense_rows_bwd(x, h, U_dense, Wg_t, Wu_t, Wd, D, dy, l1_coeff, dx, dWg_t, dWu_t, dWd,
                        w, L, status_dev, dev, s);
}

namespace twell {

twell_status dense_rows_bwd(const uint16_t* x, const hybrid_t* h, const float* U_dense,
                            const uint16_t* Wg_t, const uint16_t* Wu_t, const uint16_t* Wd,
                            int32_t D, const float* dy, float l1_coeff, float* dx, float* dWg_t,
                            float* dWu_t, float* dWd, uint8_t* w, const WsLayout& L,
                            int32_t* status_dev, const DeviceInfo& dev, cudaStream_t s) {
  const int32_t F = h->F;
  twell_status st;
  const int32_t MD = h->max_dense;
  const int64_t mp = L.mpad;
  uint16_t* Xo = reinterpret_cast<uint16_t*>(w + L.xo);
  uint16_t* dYs = reinterpret_cast<uint16_t*>(w + L.dys);
  uint16_t* G = reinterpret_cast<uint16_t*>(w + L.g);
  uint16_t* WgT = reinterpret_cast<uint16_t*>(w + L.wgT);
  uint16_t* WuT = reinterpret_cast<uint16_t*>(w + L.wuT);
  uint16_t* XoT = reinterpret_cast<uint16_t*>(w + L.xoT);
  uint16_t* dyT_hi = reinterpret_cast<uint16_t*>(w + L.dyT_hi);
  uint16_t* dyT_lo = reinterpret_cast<uint16_t*>(w + L.dyT_lo);
  uint16_t* dzT_hi = reinterpret_cast<uint16_t*>(w + L.dzT_hi);
  uint16_t* dzT_lo = reinterpret_cast<uint16_t*>(w + L.dzT_lo);
  uint16_t* duT_hi = reinterpret_cast<uint16_t*>(w + L.duT_hi);
  uint16_t* duT_lo = reinterpret_cast<uint16_t*>(w + L.duT_lo);
  uint16_t* aoT_hi = reinterpret_cast<uint16_t*>(w + L.aoT_hi);
  uint16_t* aoT_lo = reinterpret_cast<uint16_t*>(w + L.aoT_lo);
  const int64_t F64 = F, D64 = D;

  {  // dY rows split into bf16 hi | lo
    GatherArgs g{};
    g.src = dy;
    g.lds = D;
    g.row_idx = h->dense_rows;
    g.row_limit = h->T;
    g.R = MD;
    g.C = D;
    g.R_dyn = h->n_dense;
    g.out = dYs;
    g.ldo = 2 * D64;
    if ((st = gather_run(1, g, s)) != TWELL_OK) return st;
  }
  {  // W_g, W_u transposed to [D][F]
    TransposeArgs tr{};
    tr.lds = D;
    tr.R = F;
    tr.C = D;
    tr.R_pad = F;
    tr.ldo = F;
    tr.src = Wg_t;
    tr.out_hi = WgT;
    if ((st = transpose_run(0, tr, s)) != TWELL_OK) return st;
    tr.src = Wu_t;
    tr.out_hi = WuT;
    if ((st = transpose_run(0, tr, s)) != TWELL_OK) return st;
  }
  const int num_m = (MD + 127) / 128;
  {  // G3: dA = dY W_d^T -> dz, du splits in G [MD][4F]
    const bool wide = static_cast<long long>(num_m) * ((F + 255) / 256) >= dev.sm_count;
    GemmMaps maps;
    if ((st = gemm_map(&maps.a[0], dYs, MD, D, 2 * D64, false)) != TWELL_OK) return st;
    if ((st = gemm_map(&maps.a[1], dYs + D, MD, D, 2 * D64, false)) != TWELL_OK) return st;
    if ((st = gemm_map(&maps.b[0], Wd, F, D, D, wide)) != TWELL_OK) return st;
    GemmArgs a{};
    a.M = MD;
    a.N = F;
    a.M_dyn = h->n_dense;
    a.nseg = 2;
    a.seg[0] = GemmSeg{0, 0, D, nullptr};
    a.seg[1] = GemmSeg{1, 0, D, nullptr};
    a.epi = EPI_DA;
    a.H = h->dense_h;
    a.U_in = U_dense;
    a.S_out = G;
    a.lds = 4 * F64;
    a.lambda = l1_coeff;
    a.status = status_dev;
    if ((st = gemm_run(maps, a, wide, dev, s)) != TWELL_OK) return st;
  }
  {  // G4: dx[dense rows] = dz W_g^T + du W_u^T
    const bool wide = static_cast<long long>(num_m) * ((D + 255) / 256) >= dev.sm_count;
    GemmMaps maps;
    for (int q = 0; q < 4; ++q)
      if ((st = gemm_map(&maps.a[q], G + q * F64, MD, F, 4 * F64, false)) != TWELL_OK) return st;
    if ((st = gemm_map(&maps.b[0], WgT, D, F, F, wide)) != TWELL_OK) return st;
    if ((st = gemm_map(&maps.b[1], WuT, D, F, F, wide)) != TWELL_OK) return st;
    GemmArgs a{};
    a.M = MD;
    a.N = D;
    a.M_dyn = h->n_dense;
    a.nseg = 4;
    a.seg[0] = GemmSeg{0, 0, F, nullptr};
    a.seg[1] = GemmSeg{1, 0, F, nullptr};
    a.seg[2] = GemmSeg{2, 1, F, nullptr};
    a.seg[3] = GemmSeg{3, 1, F, nullptr};
    a.epi = EPI_STORE;
    a.C = dx;
    a.ldc = D;
    a.row_idx = h->dense_rows;
    a.row_limit = h->T;
    a.status = status_dev;
    a.ksplit = gemm_ksplit(static_cast<int64_t>(num_m) * ((D + (wide ? 255 : 127)) /
                                                           (wide ? 256 : 128)),
                           4 * F64, dev);
    if ((st = zero_rows(dx, D, h->dense_rows, MD, h->n_dense, D, s, h->T, status_dev)) != TWELL_OK) return st;
    if ((st = gemm_run(maps, a, wide, dev, s)) != TWELL_OK) return st;
  }
  {  // transposed operands of the weight gradients ([F or D][mpad], zero padded)
    TransposeArgs tr{};
    tr.R = MD;
    tr.R_dyn = h->n_dense;
    tr.R_pad = static_cast<int32_t>(mp);
    tr.ldo = mp;
    tr.src = x;
    tr.lds = D;
    tr.row_idx = h->dense_rows;
    tr.row_limit = h->T;
    tr.status = status_dev;
    tr.C = D;
    tr.out_hi = XoT;
    if ((st = transpose_run(0, tr, s)) != TWELL_OK) return st;
    tr.src = dy;
    tr.out_hi = dyT_hi;
    tr.out_lo = dyT_lo;
    if ((st = transpose_run(1, tr, s)) != TWELL_OK) return st;
    tr.row_idx = nullptr;
    tr.C = F;
    tr.lds = 4 * F64;
    tr.out_lo = nullptr;
    uint16_t* outs[4] = {dzT_hi, dzT_lo, duT_hi, duT_lo};
    for (int q = 0; q < 4; ++q) {
      tr.src = G + q * F64;
      tr.out_hi = outs[q];
      if ((st = transpose_run(0, tr, s)) != TWELL_OK) return st;
    }
    tr.src = U_dense;
    tr.lds = F;
    tr.src2 = h->dense_h;
    tr.lds2 = F;
    tr.out_hi = aoT_hi;
    tr.out_lo = aoT_lo;
    if ((st = transpose_run(2, tr, s)) != TWELL_OK) return st;
  }
  {  // G5-G7: weight gradients of the dense rows, added to the ELL part
    const bool wide = static_cast<long long>((F + 127) / 128) * ((D + 255) / 256) >= dev.sm_count;
    const int32_t mp32 = static_cast<int32_t>(mp);
    struct Job {
      uint16_t* a0;
      uint16_t* a1;
      uint16_t* b0;
      uint16_t* b1;
      float* C;
      bool three;
    };
    const Job jobs[3] = {{dzT_hi, dzT_lo, XoT, XoT, dWg_t, false},
                         {duT_hi, duT_lo, XoT, XoT, dWu_t, false},
                         {aoT_hi, aoT_lo, dyT_hi, dyT_lo, dWd, true}};
    for (const Job& jb : jobs) {
      GemmMaps maps;
      if ((st = gemm_map(&maps.a[0], jb.a0, F, mp, mp, false)) != TWELL_OK) return st;
      if ((st = gemm_map(&maps.a[1], jb.a1, F, mp, mp, false)) != TWELL_OK) return st;
      if ((st = gemm_map(&maps.b[0], jb.b0, D, mp, mp, wide)) != TWELL_OK) return st;
      if ((st = gemm_map(&maps.b[1], jb.b1, D, mp, mp, wide)) != TWELL_OK) return st;
      GemmArgs a{};
      a.M = F;
      a.N = D;
      a.M_dyn = nullptr;
      if (jb.three) {  // a_hi dy_hi + a_hi dy_lo + a_lo dy_hi
        a.nseg = 3;
        a.seg[0] = GemmSeg{0, 0, mp32, h->n_dense};
        a.seg[1] = GemmSeg{0, 1, mp32, h->n_dense};
        a.seg[2] = GemmSeg{1, 0, mp32, h->n_dense};
      } else {  // (hi + lo) x
        a.nseg = 2;
        a.seg[0] = GemmSeg{0, 0, mp32, h->n_dense};
        a.seg[1] = GemmSeg{1, 1, mp32, h->n_dense};
      }
      a.epi = EPI_ADD;
      a.C = jb.C;
      a.ldc = D;
      a.status = status_dev;
      if ((st = gemm_run(maps, a, wide, dev, s)) != TWELL_OK) return st;
    }
  }
  return TWELL_OK;
}

}  // namespace twell
