// K2: head-parallel chunk recurrence of the KDA chunked forward, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// One CTA per (sequence, head, 64-wide slice of V). The CTA walks the chunks
// of its sequence in order and carries its K x 64 slice of the state S (the
// FlashKDA "K2" stage, FlashKDA page, section "커널 퓨전(Kernel Fusion) 전략의
// 분리"; the cuLA "chunk gated delta h" + "chunk fwd o" stages, cuLA launch
// blog, section "Status & Roadmap"). Per chunk, with M = [-Tb ; P Tb] from
// the prep kernel and G the in-chunk cumulative decay from the chunk start:
//
//   D1 = M (khat 2^G)            = [-w ; P w]        (128 x K,  UMMA 128xKx64)
//   D2 = M v                     = [-u ; P u]        (128 x 64, UMMA 128x64x64)
//   WQ = [w ; q~ - P w],  q~ = qhat 2^G              (threads, fp16)
//   D2 += WQ S                   = [-U ; O]          (UMMA 128x64xK)
//   U -> fp16, o = scale O -> bf16                   (threads)
//   D3 = k~^T U,  k~ = khat 2^{G_last - G}           (UMMA 128x64x64)
//   S  = 2^{G_last} S + D3                           (threads, fp32 master in registers)
//
// U holds the delta-rule residuals v - prediction of the chunk, O the
// inter-chunk term q~ S plus the intra-chunk term P U. The decays 2^G and
// 2^{G_last-G} are prefix/suffix products of the per-token alpha, all <= 1.
// Operands are fp16 in shared memory (128-byte swizzled canonical layouts),
// accumulators fp32 in tensor memory; the state master copy stays fp32 in
// registers (thread k owns row k of S) and an fp16 copy feeds the next chunk.
#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {

constexpr int kRecThreads = 128;
constexpr int kBV = 64;
constexpr uint32_t kTmemCols = 256;
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clocks per wait

template <int K>
struct RecLayout {
  // byte offsets from the 1024-aligned dynamic shared memory base
  static constexpr uint32_t kPanel64 = 64 * 128;                 // 64 rows x 128 B
  static constexpr uint32_t Mh = 0;                              // 128 x 64  K-major (A of D1, D2)
  static constexpr uint32_t kG = Mh + 128 * 128;                 // 64 x K    MN-major (B of D1)
  static constexpr uint32_t vh = kG + (K / 64) * kPanel64;       // 64 x 64   MN-major (B of D2)
  static constexpr uint32_t WQ = vh + kPanel64;                  // 128 x K   K-major (A of MMA1)
  static constexpr uint32_t Sh = WQ + (K / 64) * 128 * 128;      // K x 64    MN-major (B of MMA1)
  static constexpr uint32_t kT = Sh + K * 128;                   // 64 x 128  MN-major (A of MMA2)
  static constexpr uint32_t Uh = kT + 2 * kPanel64;              // 64 x 64   MN-major (B of MMA2)
  static constexpr uint32_t qt = Uh + kPanel64;                  // fp32 [64][K]
  static constexpr uint32_t rq = qt + 64 * K * 4;               // raw bf16 q, k, g [64][K], v [64][64]
  static constexpr uint32_t rk = rq + 64 * K * 2;
  static constexpr uint32_t rg = rk + 64 * K * 2;
  static constexpr uint32_t rv = rg + 64 * K * 2;
  static constexpr uint32_t misc = rv + 64 * kBV * 2;
  static constexpr uint32_t bytes = misc + 1024 + 1024;          // + misc + alignment slack
  static_assert(64 * K * 4 <= (K / 64) * 128 * 128, "alpha scratch must fit in WQ");
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

template <int K>
__global__ void __launch_bounds__(kRecThreads, 1)
recur_tc_kernel(const Problem p) {
  using Lay = RecLayout<K>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                        ~static_cast<uintptr_t>(1023));
  float *qt = reinterpret_cast<float *>(sm + Lay::qt);
  float *alpha_s = reinterpret_cast<float *>(sm + Lay::WQ);   // per-channel pass scratch
  __nv_bfloat16 *rq = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rq);
  __nv_bfloat16 *rk = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rk);
  __nv_bfloat16 *rg = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rg);
  __nv_bfloat16 *rv = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rv);
  float *kn = reinterpret_cast<float *>(sm + Lay::misc);
  float *qn = kn + 64;
  uint64_t *bar = reinterpret_cast<uint64_t *>(qn + 64);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);
  int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int VT = p.V / kBV;
  const int bid = blockIdx.x;
  const int r = bid / (p.H * VT);
  const int h = (bid / VT) % p.H;
  const int v0 = (bid % VT) * kBV;
  if (p.flag && *p.flag != kDevOk) return;
  const int s = p.cu ? p.order[r] : r;
  const SeqInfo si = seq_info(p, s);
  const uint32_t sbase = umma::smem_u32(sm);

  // ---- set-up: zero the k~ operand (rows >= K stay zero when K = 64), TMEM, barrier
  for (int x = tid; x < (int)(2 * Lay::kPanel64 / 16); x += kRecThreads)
    reinterpret_cast<uint4 *>(sm + Lay::kT)[x] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    umma::tmem_alloc(tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    umma::mbar_init(bar, 1);
    umma::mbar_fence_init();
    *s_err = 0;
  }

  // state master: thread k owns S[k][0:64] (fp32), also written as the fp16 operand
  float S[kBV];
  if (tid < K) {
#pragma unroll
    for (int v = 0; v < kBV; ++v)
      S[v] = p.init ? p.init[(((long long)s * p.H + h) * p.V + v0 + v) * K + tid] : 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 w;
      w.x = pack_half2(S[8 * c + 0], S[8 * c + 1]);
      w.y = pack_half2(S[8 * c + 2], S[8 * c + 3]);
      w.z = pack_half2(S[8 * c + 4], S[8 * c + 5]);
      w.w = pack_half2(S[8 * c + 6], S[8 * c + 7]);
      *reinterpret_cast<uint4 *>(sm + Lay::Sh + umma::sw128_chunk(tid, c)) = w;
    }
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tD1 = tmem, tD2 = tmem + 128, tD3 = tmem + 192;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  const float ea = expf(p.A_log[h]);
  const float lbl2 = p.lb * kLog2e;
  const float dt = (tid < K && p.dt_bias) ? p.dt_bias[h * K + tid] : 0.f;
  const int nch = (si.len + kChunk - 1) / kChunk;
  uint32_t phase = 0;
  float gam = 1.f;

  // Bounded wait on the MMA barrier; every thread learns whether anyone timed out.
  auto wait_mma = [&]() -> bool {
    if (!umma::mbar_wait_bounded(bar, phase, kWaitLimit)) atomicExch(s_err, 1);
    phase ^= 1u;
    __syncthreads();
    umma::fence_after_sync();
    return *s_err == 0;
  };

  // Hand-off matrix of chunk c goes straight into its swizzled K-major operand layout.
  auto stage_mats = [&](long long c) {
    const __half *src = p.mats + (c * p.H + h) * (2 * kChunk * kChunk);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int x = tid + kRecThreads * j;   // 16-byte chunk: row x / 8, chunk x % 8
      cp_async16(sm + Lay::Mh + umma::sw128_chunk(x >> 3, x & 7), src + 8 * x, true);
    }
  };
  if (nch > 0) {
    const int L0 = min(kChunk, si.len);
    stage_rows_async<K, kRecThreads>(rq, p.q, p, si.b, si.t0, h, L0, 0, K, tid);
    stage_rows_async<K, kRecThreads>(rk, p.k, p, si.b, si.t0, h, L0, 0, K, tid);
    stage_rows_async<K, kRecThreads>(rg, p.g, p, si.b, si.t0, h, L0, 0, K, tid);
    stage_rows_async<kBV, kRecThreads>(rv, p.v, p, si.b, si.t0, h, L0, v0, p.V, tid);
    stage_mats(si.chunk0);
    cp_async_commit();
  }

  bool ok = true;
  for (int n = 0; n < nch && ok; ++n) {
    const int t0 = si.t0 + n * kChunk;
    const int L = min(kChunk, si.len - n * kChunk);

    // ---- A1: inputs of this chunk are staged (issued one chunk ahead); row norms; v tile -> fp16 operand
    cp_async_wait_all();
    __syncthreads();
    for (int i = warp; i < kChunk; i += kRecThreads / 32) {
      float ssk = 0.f, ssq = 0.f;
      const __nv_bfloat162 *kr = reinterpret_cast<const __nv_bfloat162 *>(rk + i * K);
      const __nv_bfloat162 *qr = reinterpret_cast<const __nv_bfloat162 *>(rq + i * K);
#pragma unroll
      for (int x = lane; x < K / 2; x += 32) {
        const float2 a = __bfloat1622float2(kr[x]), b = __bfloat1622float2(qr[x]);
        ssk += a.x * a.x + a.y * a.y;
        ssq += b.x * b.x + b.y * b.y;
      }
      ssk = warp_sum(ssk);
      ssq = warp_sum(ssq);
      if (lane == 0) {
        kn[i] = (i < L) ? rsqrtf(ssk + kNormEps) : 0.f;
        qn[i] = (i < L) ? rsqrtf(ssq + kNormEps) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int x = tid + kRecThreads * j;   // v tile: row x / 8, 8 values from column 8 * (x % 8)
      const int i = x >> 3, cc = x & 7;
      const uint4 raw = *reinterpret_cast<const uint4 *>(rv + i * kBV + 8 * cc);
      const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
      const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
      const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
      *reinterpret_cast<uint4 *>(sm + Lay::vh + umma::sw128_chunk(i, cc)) =
          make_uint4(pack_half2(f0.x, f0.y), pack_half2(f1.x, f1.y), pack_half2(f2.x, f2.y),
                     pack_half2(f3.x, f3.y));
    }
    __syncthreads();

    // ---- A2: per-channel gate, prefix/suffix decay products, decayed operands (thread = channel)
    if (tid < K) {
      const int kk = tid;
      const uint32_t col_off = (uint32_t)(kk >> 6) * Lay::kPanel64;
      float Gam = 1.f;
      for (int i = 0; i < kChunk; ++i) {
        float al = 1.f;
        if (i < L) al = ex2_approx(log2_decay(__bfloat162float(rg[i * K + kk]), dt, ea, lbl2));
        const float kv = __bfloat162float(rk[i * K + kk]) * kn[i];
        const float qv = __bfloat162float(rq[i * K + kk]) * qn[i];
        Gam *= al;
        alpha_s[i * K + kk] = al;
        *reinterpret_cast<__half *>(sm + Lay::kG + col_off + umma::sw128_offset(i, kk & 63)) =
            __float2half_rn(kv * Gam);
        qt[i * K + kk] = qv * Gam;
      }
      gam = Gam;
      float suf = 1.f;
      for (int i = kChunk - 1; i >= 0; --i) {
        const float kv = __bfloat162float(rk[i * K + kk]) * kn[i];
        *reinterpret_cast<__half *>(sm + Lay::kT + col_off + umma::sw128_offset(i, kk & 63)) =
            __float2half_rn(kv * suf);
        suf *= alpha_s[i * K + kk];
      }
    }
    __syncthreads();
    // raw q, k, g, v of this chunk are consumed: prefetch the next chunk's
    if (n + 1 < nch) {
      const int t1 = t0 + kChunk, L1 = min(kChunk, si.len - (n + 1) * kChunk);
      stage_rows_async<K, kRecThreads>(rq, p.q, p, si.b, t1, h, L1, 0, K, tid);
      stage_rows_async<K, kRecThreads>(rk, p.k, p, si.b, t1, h, L1, 0, K, tid);
      stage_rows_async<K, kRecThreads>(rg, p.g, p, si.b, t1, h, L1, 0, K, tid);
      stage_rows_async<kBV, kRecThreads>(rv, p.v, p, si.b, t1, h, L1, v0, p.V, tid);
      cp_async_commit();
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();

    // ---- B: D1 = M (khat 2^G), D2 = M v
    if (tid == 0) {
      umma::fence_after_sync();
      const uint32_t id1 = umma::idesc_f16(128, K, 0, 1), id2 = umma::idesc_f16(128, kBV, 0, 1);
#pragma unroll
      for (int ks = 0; ks < kChunk / 16; ++ks) {
        const uint64_t a = umma::sdesc_sw128(sbase + Lay::Mh + ks * 32, 16, 1024);
        umma::mma_f16_ss(tD1, a, umma::sdesc_sw128(sbase + Lay::kG + ks * 2048, Lay::kPanel64, 1024), id1, ks > 0);
        umma::mma_f16_ss(tD2, a, umma::sdesc_sw128(sbase + Lay::vh + ks * 2048, Lay::kPanel64, 1024), id2, ks > 0);
      }
      umma::commit(bar);
    }
    if (!(ok = wait_mma())) break;
    if (n + 1 < nch) {   // M is consumed by D1/D2: prefetch the next chunk's
      stage_mats((long long)si.chunk0 + n + 1);
      cp_async_commit();
    }

    // ---- C: WQ rows: w = -D1 (rows < 64), Q' = q~ - D1 (rows >= 64)
#pragma unroll 1
    for (int c0 = 0; c0 < K; c0 += 16) {
      float x[16];
      umma::tmem_ld16(tD1 + lane_base + c0, x);
      umma::tmem_ld_wait();
      if (tid < kChunk) {
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = -x[j];
      } else {
        const float *qr = qt + (tid - kChunk) * K + c0;
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = qr[j] - x[j];
      }
      const uint32_t pan = Lay::WQ + (uint32_t)(c0 >> 6) * (128 * 128);
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        uint4 w;
        w.x = pack_half2(x[8 * hc + 0], x[8 * hc + 1]);
        w.y = pack_half2(x[8 * hc + 2], x[8 * hc + 3]);
        w.z = pack_half2(x[8 * hc + 4], x[8 * hc + 5]);
        w.w = pack_half2(x[8 * hc + 6], x[8 * hc + 7]);
        *reinterpret_cast<uint4 *>(sm + pan + umma::sw128_chunk(tid, ((c0 & 63) >> 3) + hc)) = w;
      }
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();

    // ---- D: D2 += WQ S  ->  [-U ; O]
    if (tid == 0) {
      umma::fence_after_sync();
      const uint32_t id = umma::idesc_f16(128, kBV, 0, 1);
#pragma unroll
      for (int ks = 0; ks < K / 16; ++ks) {
        const uint64_t a = umma::sdesc_sw128(sbase + Lay::WQ + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
        const uint64_t b = umma::sdesc_sw128(sbase + Lay::Sh + ks * 2048, K * 128, 1024);
        umma::mma_f16_ss(tD2, a, b, id, 1);
      }
      umma::commit(bar);
    }
    if (!(ok = wait_mma())) break;

    // ---- E: U (rows < 64) -> fp16 operand; o = scale * O (rows >= 64) -> bf16 global
#pragma unroll 1
    for (int c0 = 0; c0 < kBV; c0 += 16) {
      float x[16];
      umma::tmem_ld16(tD2 + lane_base + c0, x);
      umma::tmem_ld_wait();
      if (tid < kChunk) {
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          uint4 w;
          w.x = pack_half2(-x[8 * hc + 0], -x[8 * hc + 1]);
          w.y = pack_half2(-x[8 * hc + 2], -x[8 * hc + 3]);
          w.z = pack_half2(-x[8 * hc + 4], -x[8 * hc + 5]);
          w.w = pack_half2(-x[8 * hc + 6], -x[8 * hc + 7]);
          *reinterpret_cast<uint4 *>(sm + Lay::Uh + umma::sw128_chunk(tid, (c0 >> 3) + hc)) = w;
        }
      } else if (tid - kChunk < L) {
        __nv_bfloat16 ob[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) ob[j] = __float2bfloat16_rn(p.scale * x[j]);
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + tok_row(p, si.b, t0 + tid - kChunk, h) * p.V + v0 + c0);
        dst[0] = *reinterpret_cast<const uint4 *>(&ob[0]);
        dst[1] = *reinterpret_cast<const uint4 *>(&ob[8]);
      }
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();

    // ---- F: D3 = k~^T U
    if (tid == 0) {
      umma::fence_after_sync();
      const uint32_t id = umma::idesc_f16(128, kBV, 1, 1);
#pragma unroll
      for (int ks = 0; ks < kChunk / 16; ++ks) {
        const uint64_t a = umma::sdesc_sw128(sbase + Lay::kT + ks * 2048, Lay::kPanel64, 1024);
        const uint64_t b = umma::sdesc_sw128(sbase + Lay::Uh + ks * 2048, Lay::kPanel64, 1024);
        umma::mma_f16_ss(tD3, a, b, id, ks > 0);
      }
      umma::commit(bar);
    }
    if (!(ok = wait_mma())) break;

    // ---- G: S = gamma S + D3 (thread = channel), fp16 copy for the next chunk
    if (tid < K) {
#pragma unroll
      for (int c0 = 0; c0 < kBV; c0 += 16) {
        float x[16];
        umma::tmem_ld16(tD3 + lane_base + c0, x);
        umma::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) S[c0 + j] = fmaf(gam, S[c0 + j], x[j]);
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          uint4 w;
          const float *sv = &S[c0 + 8 * hc];
          w.x = pack_half2(sv[0], sv[1]);
          w.y = pack_half2(sv[2], sv[3]);
          w.z = pack_half2(sv[4], sv[5]);
          w.w = pack_half2(sv[6], sv[7]);
          *reinterpret_cast<uint4 *>(sm + Lay::Sh + umma::sw128_chunk(tid, (c0 >> 3) + hc)) = w;
        }
      }
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
  }

  cp_async_wait_all();
  if (!ok) {
    if (tid == 0) atomicExch(p.dev_status, kDevWaitTimeout);
    // one more bounded wait (on the phase that timed out) so that no MMA of
    // this CTA is still writing TMEM when it is released
    umma::mbar_wait_bounded(bar, phase ^ 1u, kWaitLimit);
  } else if (p.final_state && tid < K) {
#pragma unroll
    for (int v = 0; v < kBV; ++v) p.final_state[(((long long)s * p.H + h) * p.V + v0 + v) * K + tid] = S[v];
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

template <int K>
static cudaError_t launch_recur_t(const Problem &p, cudaStream_t stream) {
  const size_t smem = RecLayout<K>::bytes;
  cudaError_t e = cudaFuncSetAttribute(recur_tc_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.H * (p.V / kBV);
  recur_tc_kernel<K><<<(unsigned)grid, kRecThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_recur(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  return p.K == 64 ? launch_recur_t<64>(p, stream) : launch_recur_t<128>(p, stream);
}

}  // namespace kda
