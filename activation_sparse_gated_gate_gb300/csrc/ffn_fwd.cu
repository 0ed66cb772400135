// Fused up + down projection driven by the TwELL gate ("Sparser, Faster,
// Lighter Transformer Language Models", section 2.B.2: one kernel does the
// up and down projections from the TwELL gate activations, computing dot
// products only for the nonzero elements and keeping DRAM traffic low).
//
// Work unit = (token row t, range of G column tiles); one warp per unit at a
// time (12 warps per CTA for D <= 2304, else 8; one CTA per SM).  With
// many tokens G covers the whole row and the warp stores y_t; with few
// tokens (decode) rows are split into several units so every SM gets work,
// and each unit adds its partial y_t with 16-byte atomics into a zeroed y.
// Each CTA takes a contiguous range of units and hands them to its warps in
// order of completion.
// x_t (bf16 pairs) and the fp32 accumulator of y_t live in registers, spread
// over the 32 lanes in 8-element chunks (lane l holds chunks l, l+32, ...).
//
// Per unit the warp first lists its active entries (j, h) in shared memory:
// the counts of 32 tiles are read at once, a warp prefix sum places every
// tile's entries, and each lane copies its tile's slots (or scans its spill
// slice).  The warp then walks the list through a ring of P shared-memory
// stages: lane 0 issues two cp.async.bulk copies per entry (neuron j's rows
// W_u^T[j] and W_d[j], 2*D contiguous bf16 each) completing on the stage's
// mbarrier, P entries ahead of the compute.  Per entry the lanes read the
// staged rows with 16-byte shared loads, form u = x_t . W_u[:, j] with the
// mixed-precision FMA (bf16 x bf16 products into eight independent fp32
// sums: x_t and W_u stay bf16, nothing is widened) and a butterfly
// reduction, and accumulate (h u) W_d[j, :] with the packed fp32-pair FMA
// (fma.rn.f32x2) on W_d's bf16 pairs widened to fp32 pairs.
#include "bounds.cuh"
#include "fused.cuh"
#include "ptx.cuh"

namespace twell {
namespace {

constexpr int kListCap = 64;         // entries listed per pass

// Warps per CTA (one CTA per SM): 12 while a thread's row state fits in
// 65536 / 384 registers without spills (D <= 2304), else 8.  Measured with
// CUDA events: 0.5B-class shape 324 -> 271 us, 1.5B-class 1377 -> 1123 us,
// 2B-class ELL forward 4.13 -> 3.35 ms against 8 warps.
__host__ __device__ constexpr int warps_for(int nc) { return nc <= 9 ? 12 : 8; }
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 231168;  // within the 227 KB opt-in limit

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

// lo += a.lo * b.lo, hi += a.hi * b.hi on bf16 pairs: bf16 x bf16 products,
// fp32 addends and results (mixed-precision FMA)
__device__ __forceinline__ void dot_bf16x2(float& lo, float& hi, uint32_t a, uint32_t b) {
  asm("{\n"
      ".reg .b16 al, ah, bl, bh;\n"
      "mov.b32 {al, ah}, %2;\n"
      "mov.b32 {bl, bh}, %3;\n"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n"
      "fma.rn.f32.bf16 %1, ah, bh, %1;\n"
      "}\n"
      : "+f"(lo), "+f"(hi)
      : "r"(a), "r"(b));
}

// NC = 8-element chunks per lane (D <= 256 * NC).  EXACT: D == 256 * NC, so
// every lane owns all NC of its chunks.
template <int NC, bool EXACT, bool ELL>
__global__ void __launch_bounds__(warps_for(NC) * 32, 1) ffn_fwd_kernel(const FfnParams p) {
  constexpr int kWarps = warps_for(NC);
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int P = p.stages;
  const int D = p.D;
  const int nch = D >> 3;
  const uint32_t row_bytes = static_cast<uint32_t>(D) * 2u;

  uint8_t* wbase = smem + static_cast<size_t>(wid) * p.warp_bytes;
  uint8_t* stages = wbase;                                   // P x [W_u row | W_d row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + static_cast<size_t>(P) * 2 * row_bytes);
  Entry* list = reinterpret_cast<Entry*>(bars + kMaxStages);

  if (lane == 0) {
    for (int s = 0; s < P; ++s) ptx::mbar_init(&bars[s], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  auto own = [&](int i) { return EXACT || (lane + 32 * i) < nch; };
  uint32_t seq = 0;  // entries issued (and consumed) so far by this warp

  auto issue = [&](const Entry& e, uint32_t n) {
    const int s = static_cast<int>(n % static_cast<uint32_t>(P));
    uint8_t* dst = stages + static_cast<size_t>(s) * 2 * row_bytes;
    const size_t j = static_cast<size_t>(
        clamp_index(e.j, static_cast<long long>(p.n_t) * TWELL_TILE, p.status));
    ptx::mbar_arrive_expect_tx(&bars[s], 2 * row_bytes);
    ptx::bulk_load(dst, p.Wu_t + j * D, row_bytes, &bars[s]);
    ptx::bulk_load(dst + row_bytes, p.Wd + j * D, row_bytes, &bars[s]);
  };

  // Each CTA owns a contiguous range of units; its warps take the next unit
  // of the range from a shared counter as they finish the previous one, so a
  // few heavy rows delay one warp by one row rather than a fixed share.
  __shared__ int next_unit;
  const long long units =
      ELL ? static_cast<long long>(*p.n_rows) : static_cast<long long>(p.T) * p.upr;
  const long long u_begin = units * blockIdx.x / gridDim.x;
  const long long u_end = units * (blockIdx.x + 1) / gridDim.x;
  if (threadIdx.x == 0) next_unit = 0;
  __syncthreads();
  for (;;) {
    int take = 0;
    if (lane == 0) take = atomicAdd(&next_unit, 1);
    const long long u = u_begin + __shfl_sync(0xffffffffu, take, 0);
    if (u >= u_end) break;
    // row: index into the count / slot arrays; t: token (x and y row)
    const int row = ELL ? static_cast<int>(u) : static_cast<int>(u / p.upr);
    const int t = ELL ? p.ell_rows[row] : row;
    if (ELL && !in_bounds(t, p.T, p.status)) continue;  // warp-uniform
    const int k_begin = static_cast<int>(u % p.upr) * p.G;
    const int k_end = min(k_begin + p.G, p.n_t);
    uint32_t xb[NC][4];
    float acc[NC][8];
    bool any = false;
    const uint16_t* xr = p.x + static_cast<size_t>(t) * D;
    // x_t is loaded at once, with the counts and slots below in flight, not
    // after them (at decode sizes every dependent load is a DRAM round trip)
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      const uint4 v = own(i) ? __ldg(reinterpret_cast<const uint4*>(xr + 8 * (lane + 32 * i)))
                             : make_uint4(0, 0, 0, 0);
      xb[i][0] = v.x;
      xb[i][1] = v.y;
      xb[i][2] = v.z;
      xb[i][3] = v.w;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] = 0.0f;
    }

    const size_t row_rt = static_cast<size_t>(row) * p.n_t;
    for (int kb = k_begin; kb < k_end; kb += 32) {
      const int k = kb + lane;
      int c = k < k_end ? p.cnt[row_rt + k] : 0;
      // the tile's first four slots, loaded beside its count (used below
      // when the count is known; read past the count, never used there)
      const bool pre = (p.W & 3) == 0 && k < k_end;
      const size_t so_k = (row_rt + k) * static_cast<size_t>(p.W);
      const float4 v_pre =
          pre ? __ldg(reinterpret_cast<const float4*>(p.val + so_k)) : make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t c_pre = pre ? __ldg(reinterpret_cast<const uint32_t*>(p.col + so_k)) : 0u;
      if (!in_bounds(c, (ELL ? p.W : TWELL_TILE) + 1, p.status)) c = 0;
      // entries of tile k: its slots, or the positives of its spill slice
      // (the spill holds exactly c positive values)
      int spill = -1;
      if (!ELL && c > p.W) {
        spill = p.spill_slot[row_rt + k];
        if (spill < 0 || spill >= p.spill_cap) {
          atomicOr(p.status, TWELL_FLAG_SPILL_FULL);
          spill = -2;
        }
      }
      const int n = spill == -2 ? 0 : c;
      int off = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, off, d);
        if (lane >= d) off += v;
      }
      const int total = __shfl_sync(0xffffffffu, off, 31);
      off -= n;
      any |= total > 0;

      for (int base = 0; base < total; base += kListCap) {
        // list the entries whose position falls in [base, base + kListCap)
        if (n > 0 && off + n > base && off < base + kListCap) {
          const int jbase = k * TWELL_TILE;
          if (spill < 0) {
            const size_t so = (row_rt + k) * static_cast<size_t>(p.W);
            const int s0 = max(0, base - off);
            const int s1 = min(n, base + kListCap - off);
            if ((p.W & 3) == 0) {
              // four slots per 16-byte load (slots past the count are read, not used)
              for (int q = s0 & ~3; q < s1; q += 4) {
                const float4 v =
                    q == 0 ? v_pre : __ldg(reinterpret_cast<const float4*>(p.val + so + q));
                const uint32_t c4 =
                    q == 0 ? c_pre : __ldg(reinterpret_cast<const uint32_t*>(p.col + so + q));
                const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int s = q + e;
                  if (s >= s0 && s < s1)
                    list[off + s - base] = Entry{jbase + tile_col((c4 >> (8 * e)) & 0xffu),
                                                 vv[e], static_cast<int32_t>(so + s)};
                }
              }
            } else {
              for (int s = s0; s < s1; ++s)
                list[off + s - base] =
                    Entry{jbase + tile_col(p.col[so + s]), p.val[so + s], static_cast<int32_t>(so + s)};
            }
          } else {
            const float* sl = p.spill_val + static_cast<size_t>(spill) * TWELL_TILE;
            int e = off;
            for (int cc = 0; cc < TWELL_TILE && e < base + kListCap; ++cc) {
              const float v = sl[cc];
              if (v > 0.0f) {
                if (e >= base) list[e - base] = Entry{jbase + cc, v, 0};
                ++e;
              }
            }
          }
        }
        __syncwarp();
        const int m = min(kListCap, total - base);
        if (lane == 0) {
          const int pre = min(P, m);
          for (int i = 0; i < pre; ++i) issue(list[i], seq + i);
        }
        for (int i = 0; i < m; ++i) {
          const uint32_t n_i = seq + i;
          const int s = static_cast<int>(n_i % static_cast<uint32_t>(P));
          // warp-uniform decision: the lanes shuffle together below
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bars[s], (n_i / P) & 1u))) {
            // before leaving, wait (bounded) for the row copies this warp
            // still has in flight into its stages: entries i .. i + P - 1
            if (lane == 0) {
              atomicOr(p.status, TWELL_FLAG_TIMEOUT);
              for (int r = i; r < min(m, i + P); ++r) {
                const uint32_t n_r = seq + r;
                if (!ptx::mbar_wait(&bars[n_r % static_cast<uint32_t>(P)], (n_r / P) & 1u)) break;
              }
            }
            __syncwarp();
            return;
          }
          const Entry e = list[i];
          const uint4* su =
              reinterpret_cast<const uint4*>(stages + static_cast<size_t>(s) * 2 * row_bytes);
          const uint4* sd = su + nch;
          float pp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < NC; ++q) {
            if (own(q)) {
              const uint4 a = su[lane + 32 * q];
              const uint32_t a4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
              for (int r = 0; r < 4; ++r) dot_bf16x2(pp[2 * r], pp[2 * r + 1], xb[q][r], a4[r]);
            }
          }
          float part = ((pp[0] + pp[1]) + (pp[2] + pp[3])) + ((pp[4] + pp[5]) + (pp[6] + pp[7]));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
          if (ELL && lane == 0 &&
              in_bounds(e.pos, static_cast<long long>(p.T) * p.n_t * p.W, p.status))
            p.u_save[e.pos] = part;
          const float sc = e.h * part;
          const f32x2 sc2 = pack2(sc, sc);
#pragma unroll
          for (int q = 0; q < NC; ++q) {
            if (own(q)) {
              const uint4 b = sd[lane + 32 * q];
              const uint32_t b4[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                f32x2 a2 = pack2(acc[q][2 * r], acc[q][2 * r + 1]);
                fma2(a2, sc2, pack2(bf16lo(b4[r]), bf16hi(b4[r])));
                unpack2(a2, acc[q][2 * r], acc[q][2 * r + 1]);
              }
            }
          }
          // every lane is done reading stage s before it is refilled
          __syncwarp();
          if (lane == 0 && i + P < m) {
            ptx::fence_proxy_async_smem();
            issue(list[i + P], n_i + P);
          }
        }
        seq += static_cast<uint32_t>(m);
        __syncwarp();  // the list is rewritten by the next pass
      }
    }

    float* yr = p.y + static_cast<size_t>(t) * D;
    if (p.split) {
      if (any) {
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          if (own(i)) {
            float4* o = reinterpret_cast<float4*>(yr + 8 * (lane + 32 * i));
            atomicAdd(o, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
            atomicAdd(o + 1, make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]));
          }
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        if (own(i)) {
          float4* o = reinterpret_cast<float4*>(yr + 8 * (lane + 32 * i));
          o[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
          o[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
      }
    }
  }
}

template <int NC, bool ELL>
twell_status launch_nc(FfnParams p, const DeviceInfo& dev, cudaStream_t s) {
  constexpr int kWarps = warps_for(NC);
  const int stage_bytes = 4 * p.D;
  const int fixed = kMaxStages * 8 + kListCap * static_cast<int>(sizeof(Entry));
  const int budget = kSmemBudget < dev.max_smem_optin ? kSmemBudget : dev.max_smem_optin;
  int P = (budget / kWarps - fixed) / stage_bytes;
  if (P > kMaxStages) P = kMaxStages;
  if (P < 1) return TWELL_ERR_UNSUPPORTED;
  p.stages = P;
  p.warp_bytes = (P * stage_bytes + fixed + 15) & ~15;
  const int smem = kWarps * p.warp_bytes;
  const bool exact = p.D == 256 * NC;
  auto kern = exact ? ffn_fwd_kernel<NC, true, ELL> : ffn_fwd_kernel<NC, false, ELL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return TWELL_ERR_CUDA;
  // Whole rows per unit when there are enough rows to fill every warp a few
  // times over; otherwise split rows into tile ranges, about one unit per
  // warp (each unit adds a whole partial y row with atomics, so finer splits
  // cost more atomics than they gain in parallelism: measured on the decode
  // shapes, d_model 2048, 0.5 % active, T = 64 / 256: 22.1 / 34.4 us with
  // four units per warp, 20.1 / 27.2 us with one).
  // The units per row are chosen first, at most warps / T, so no warp gets a
  // second unit (T = 256: 8 units of 8 tiles per row, 2048 units for 1824
  // warps, left warps with two units and the SMs active 19.5 k to 34.7 k
  // cycles; 7 units of at most 10 tiles give 1792).
  const long long warps_total = static_cast<long long>(dev.sm_count) * kWarps;
  if (ELL || p.T >= 4 * warps_total) {
    p.G = p.n_t;
  } else {
    const long long per_row = warps_total / p.T;
    const long long upr = per_row < 1 ? 1 : (per_row > p.n_t ? p.n_t : per_row);
    p.G = static_cast<int>((p.n_t + upr - 1) / upr);
  }
  p.upr = (p.n_t + p.G - 1) / p.G;
  p.split = p.upr > 1;
  if (p.split && !p.y_zeroed &&
      cudaMemsetAsync(p.y, 0, static_cast<size_t>(p.T) * p.D * sizeof(float), s) != cudaSuccess)
    return TWELL_ERR_CUDA;
  const long long units = static_cast<long long>(p.T) * p.upr;
  const long long want = (units + kWarps - 1) / kWarps;
  const int grid = static_cast<int>(want < dev.sm_count ? want : dev.sm_count);
  kern<<<grid, kWarps * 32, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? TWELL_OK : TWELL_ERR_CUDA;
}

}  // namespace

twell_status launch_fused(const FfnParams& p, const DeviceInfo& dev, cudaStream_t s, bool ell) {
#define TWELL_NC_CASE(n) \
  case n:                \
    return ell ? launch_nc<n, true>(p, dev, s) : launch_nc<n, false>(p, dev, s);
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

}  // namespace twell

extern "C" twell_status twell_ffn_fwd(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                                      const uint16_t* Wd, int32_t D, float* y,
                                      int32_t* status_dev, void* stream) {
  return twell::ffn_fwd_twell(x, h, Wu_t, Wd, D, y, status_dev,
                              static_cast<cudaStream_t>(stream), false);
}

namespace twell {

twell_status ffn_fwd_twell(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                           const uint16_t* Wd, int32_t D, float* y, int32_t* status_dev,
                           cudaStream_t stream, bool y_zeroed) {
  if (h == nullptr) return TWELL_ERR_INVALID;
  const int32_t T = h->T, F = h->F;
  if (T < 0 || F <= 0 || F % TWELL_TILE != 0 || D <= 0 || D % 8 != 0) return TWELL_ERR_INVALID;
  twell_status st = check_twell(h, T, F, false);
  if (st != TWELL_OK) return st;
  if (T == 0) return TWELL_OK;
  if (!x || !Wu_t || !Wd || !y || !status_dev) return TWELL_ERR_INVALID;
  if (!aligned16(x) || !aligned16(Wu_t) || !aligned16(Wd) || !aligned16(y))
    return TWELL_ERR_INVALID;
  if (D > 256 * 12) return TWELL_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if ((st = require_sm103(&dev)) != TWELL_OK) return st;

  FfnParams p;
  p.x = x;
  p.Wu_t = Wu_t;
  p.Wd = Wd;
  p.y = y;
  p.val = h->val;
  p.col = h->col;
  p.cnt = h->cnt;
  p.spill_slot = h->spill_slot;
  p.spill_val = h->spill_val;
  p.spill_cap = h->spill_cap;
  p.T = T;
  p.D = D;
  p.n_t = F / TWELL_TILE;
  p.W = h->width;
  p.status = status_dev;
  p.n_rows = nullptr;
  p.ell_rows = nullptr;
  p.u_save = nullptr;
  p.y_zeroed = y_zeroed ? 1 : 0;
  return launch_fused(p, dev, stream, false);
}

}  // namespace twell
