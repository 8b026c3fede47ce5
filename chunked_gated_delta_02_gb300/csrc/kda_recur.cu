// K2: head-parallel chunk recurrence of the KDA chunked forward, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// One CTA per (sequence, head, 64-wide slice of V). The CTA walks the chunks
// of its sequence in order and carries its K x 64 slice of the state S (the
// FlashKDA "K2" stage, FlashKDA page, section "커널 퓨전(Kernel Fusion) 전략의
// 분리"; the cuLA "chunk gated delta h" + "chunk fwd o" stages, cuLA launch
// blog, section "Status & Roadmap"). Per chunk, with M = [-Tb ; P Tb] from
// the prep kernel and the in-chunk decays measured from the chunk start:
//
//   D1 = M (khat Gamma)          = [-w ; P w]        (128 x K,  UMMA 128xKx64)
//   D2 = M v                     = [-u ; P u]        (128 x 64, UMMA 128x64x64)
//   WQ = [w ; q~ - P w],  q~ = qhat Gamma            (fp16 operand)
//   D2 += WQ S                   = [-U ; O]          (UMMA 128x64xK)
//   U -> fp16, o = scale O -> bf16
//   D3 = k~^T U,  k~ = khat Gamma_last / Gamma       (UMMA 128x64x64)
//   S  = Gamma_last S + D3                           (fp32 master in registers)
//
// Gamma_i is the product of the per-token decays alpha up to token i (all
// factors <= 1, formed as products, never as quotients). U holds the
// delta-rule residuals v - prediction of the chunk; O the inter-chunk term
// q~ S plus the intra-chunk term P U.
//
// Warp roles (the S-independent work of chunk n+1 overlaps the state chain of
// chunk n):
//   chain group, warps 0-3: D2 += WQ S, U and o, D3 = k~^T U, S update.
//   prep group, warps 4-11: stages the chunk inputs with TMA, computes
//     the gate, the decay products and the fp16 operands (one thread per
//     channel pair and 16-row block), issues D1 and D2, and forms WQ and k~.
// The groups hand over through mbarriers. Every wait gives up after a bounded
// time; the groups then agree (barrier with OR-reduction) to stop, drain their
// tensor-core work, free TMEM and report KDA_DEVICE_WAIT_TIMEOUT.
#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {

constexpr int kChainThreads = 128;
constexpr int kPrepGroupThreads = 256;
constexpr int kRecThreads = kChainThreads + kPrepGroupThreads;
constexpr int kBV = 64;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clocks per wait
constexpr int kBarPrep = 1, kBarChain = 2;        // named barrier ids (0 is __syncthreads)

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
  static constexpr uint32_t qt = Uh + kPanel64;                  // fp16 [64][K] plain
  static constexpr uint32_t rq = qt + 64 * K * 2;                // raw bf16 q, k, fp16 la2 [64][K], bf16 v [64][64]
  static constexpr uint32_t rk = rq + 64 * K * 2;
  static constexpr uint32_t rg = rk + 64 * K * 2;
  static constexpr uint32_t rv = rg + 64 * K * 2;
  static constexpr uint32_t misc = rv + 64 * kBV * 2;
  static constexpr uint32_t bytes = misc + 4096 + 1024;          // + misc + alignment slack
};

// Small per-CTA state after the operand buffers.
template <int K>
struct RecMisc {
  uint64_t bar_d12, bar_wq_full, bar_mma1, bar_mma2, bar_exit, bar_in, bar_m;
  uint32_t tmem_slot;
  int err;
  float kn[kChunk], qn[kChunk];
  float btot[4][K];          // per 16-row block and channel: product of alpha over the block
  float gam[2][K];           // per chunk (double-buffered): product of alpha over the chunk
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

template <int K>
__global__ void __launch_bounds__(kRecThreads, 1)
recur_tc_kernel(const Problem p, const __grid_constant__ TmaMaps maps) {
  using Lay = RecLayout<K>;
  constexpr int CPT = K / 64;   // channels per prep thread
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so that the
  // compiler keeps every access in the shared address space
  unsigned char *sm = smem_raw + ((1024u - (umma::smem_u32(smem_raw) & 1023u)) & 1023u);
  __half *qt = reinterpret_cast<__half *>(sm + Lay::qt);
  __nv_bfloat16 *rq = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rq);
  __nv_bfloat16 *rk = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rk);
  __nv_bfloat16 *rg = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rg);
  __nv_bfloat16 *rv = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rv);
  RecMisc<K> &ms = *reinterpret_cast<RecMisc<K> *>(sm + Lay::misc);

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
  const int nch = (si.len + kChunk - 1) / kChunk;
  const bool is_chain = warp < 4;
  const int pt = tid - kChainThreads;   // prep thread index (prep group only)

  // ---- set-up: zero the k~ operand (rows >= K stay zero when K = 64), TMEM, barriers
  for (int x = tid; x < (int)(2 * Lay::kPanel64 / 16); x += kRecThreads)
    reinterpret_cast<uint4 *>(sm + Lay::kT)[x] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    umma::tmem_alloc(&ms.tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    umma::mbar_init(&ms.bar_d12, 1);
    umma::mbar_init(&ms.bar_wq_full, 1);
    umma::mbar_init(&ms.bar_mma1, 1);
    umma::mbar_init(&ms.bar_mma2, 1);
    umma::mbar_init(&ms.bar_exit, 2);
    umma::mbar_init(&ms.bar_in, 1);
    umma::mbar_init(&ms.bar_m, 1);
    umma::mbar_fence_init();
    ms.err = 0;
  }
  // chain threads: state master S[k][0:64] (fp32, thread k) and its fp16 operand copy
  float S[kBV];
  if (is_chain && tid < K) {
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
  // Inputs of chunk n: one tiled TMA copy per tensor (q, k, g: 64 x K; v: 64 x 64 at column v0),
  // issued by one prep thread and completing on bar_in. Tokens past T read as zeros; tokens of
  // the next packed sequence are zeroed after arrival.
  auto stage_inputs = [&](int n) {
    if (pt == 0) {
      const int tn = si.t0 + n * kChunk;
      umma::mbar_arrive_expect_tx(&ms.bar_in, (uint32_t)kChunk * (3 * K * 2 + kBV * 2));
      umma::tma_load_4d(rq, &maps.q, 0, h, tn, si.b, &ms.bar_in);
      umma::tma_load_4d(rk, &maps.k, 0, h, tn, si.b, &ms.bar_in);
      umma::tma_load_4d(rg, &maps.la2, 0, h, tn, si.b, &ms.bar_in);
      umma::tma_load_4d(rv, &maps.v, v0, h, tn, si.b, &ms.bar_in);
    }
  };
  // Hand-off matrix of chunk n: stored pre-swizzled, so one 16 KB bulk copy places it.
  auto stage_mats = [&](int n) {
    if (pt == 0) {
      umma::mbar_arrive_expect_tx(&ms.bar_m, 2 * kChunk * kChunk * 2);
      umma::bulk_g2s(sm + Lay::Mh, p.mats + (((long long)si.chunk0 + n) * p.H + h) * (2 * kChunk * kChunk),
                     2 * kChunk * kChunk * 2, &ms.bar_m);
    }
  };
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (!is_chain && nch > 0) {
    stage_inputs(0);
    stage_mats(0);
  }
  const uint32_t tmem = ms.tmem_slot;
  const uint32_t tD1 = tmem, tD3 = tmem + 256;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool bad = false;   // this thread saw a wait time out
  uint32_t in_done = 0, m_done = 0;   // completed bar_in / bar_m phases seen by this thread

  auto wait_bar = [&](uint64_t *bar, uint32_t parity) {
    if (bad) return;
    if (!umma::mbar_wait_bounded(bar, parity, kWaitLimit)) {
      atomicExch(&ms.err, 1);
      bad = true;
      return;
    }
    umma::fence_after_sync();
  };

  if (is_chain) {
    // ======================= chain group =======================
    for (int n = 0; n < nch; ++n) {
      if (umma::bar_red_or(kBarChain, kChainThreads, bad || *(volatile int *)&ms.err != 0)) break;
      const uint32_t par = (uint32_t)(n & 1);
      const uint32_t tD2 = tmem + 128 + 64 * (n & 1);
      const int t0 = si.t0 + n * kChunk;
      const int L = min(kChunk, si.len - n * kChunk);
      wait_bar(&ms.bar_wq_full, par);
      const float gam = (tid < K) ? ms.gam[n & 1][tid] : 0.f;   // read before MMA1: the slot is reused
      if (tid == 0 && !bad) {   // D2 += WQ S  ->  [-U ; O]
        const uint32_t id = umma::idesc_f16(128, kBV, 0, 1);
#pragma unroll
        for (int ks = 0; ks < K / 16; ++ks) {
          const uint64_t a = umma::sdesc_sw128(sbase + Lay::WQ + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
          const uint64_t b = umma::sdesc_sw128(sbase + Lay::Sh + ks * 2048, K * 128, 1024);
          umma::mma_f16_ss(tD2, a, b, id, 1);
        }
        umma::commit(&ms.bar_mma1);
      }
      wait_bar(&ms.bar_mma1, par);
      // U (rows < 64) -> fp16 operand; o = scale * O (rows >= 64) -> bf16 global
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
        } else if (tid - kChunk < L && !bad) {
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
      umma::named_bar(kBarChain, kChainThreads);
      if (tid == 0 && !bad) {   // D3 = k~^T U
        umma::fence_after_sync();
        const uint32_t id = umma::idesc_f16(128, kBV, 1, 1);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
          const uint64_t a = umma::sdesc_sw128(sbase + Lay::kT + ks * 2048, Lay::kPanel64, 1024);
          const uint64_t b = umma::sdesc_sw128(sbase + Lay::Uh + ks * 2048, Lay::kPanel64, 1024);
          umma::mma_f16_ss(tD3, a, b, id, ks > 0);
        }
        umma::commit(&ms.bar_mma2);
      }
      wait_bar(&ms.bar_mma2, par);
      // S = gamma S + D3 (thread = channel), fp16 copy for the next chunk
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
      umma::named_bar(kBarChain, kChainThreads);
    }
  } else {
    // ======================= prep group =======================
    const int cg = pt % 64, J = pt / 64;          // channels [cg*CPT, cg*CPT+CPT), rows [16J, 16J+16)
    const uint32_t col_panel = (uint32_t)((cg * CPT) >> 6) * Lay::kPanel64;
    const int col_in = (cg * CPT) & 63;
    for (int n = 0; n < nch; ++n) {
      const uint32_t par = (uint32_t)(n & 1);
      const uint32_t tD2 = tmem + 128 + 64 * (n & 1);
      const int L = min(kChunk, si.len - n * kChunk);
      wait_bar(&ms.bar_in, par);
      in_done += bad ? 0u : 1u;
      if (L < kChunk) {   // rows past the sequence end (next packed sequence or zero fill): zero them
        for (int x = pt; x < (kChunk - L) * (3 * K + kBV) / 8; x += kPrepGroupThreads) {
          const int per_row = (3 * K + kBV) / 8, i = L + x / per_row, c = x % per_row;
          __nv_bfloat16 *dst = (c < K / 8) ? rq + i * K + 8 * c
                               : (c < 2 * K / 8) ? rk + i * K + 8 * (c - K / 8)
                               : (c < 3 * K / 8) ? rg + i * K + 8 * (c - 2 * K / 8)
                                                 : rv + i * kBV + 8 * (c - 3 * K / 8);
          *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
      }
      if (umma::bar_red_or(kBarPrep, kPrepGroupThreads, bad || *(volatile int *)&ms.err != 0)) break;
      // -- row norms: 4 threads per row, K/4 channels each (bf16x2 from the staged rows)
      {
        const int row = pt >> 2, qd = pt & 3;
        const __nv_bfloat162 *kr = reinterpret_cast<const __nv_bfloat162 *>(rk + row * K) + qd * (K / 8);
        const __nv_bfloat162 *qr = reinterpret_cast<const __nv_bfloat162 *>(rq + row * K) + qd * (K / 8);
        float ssk = 0.f, ssq = 0.f;
#pragma unroll
        for (int x = 0; x < K / 8; ++x) {
          const float2 a = __bfloat1622float2(kr[x]), b = __bfloat1622float2(qr[x]);
          ssk += a.x * a.x + a.y * a.y;
          ssq += b.x * b.x + b.y * b.y;
        }
        ssk += __shfl_xor_sync(0xffffffffu, ssk, 1);
        ssk += __shfl_xor_sync(0xffffffffu, ssk, 2);
        ssq += __shfl_xor_sync(0xffffffffu, ssq, 1);
        ssq += __shfl_xor_sync(0xffffffffu, ssq, 2);
        if (qd == 0) {
          ms.kn[row] = (row < L) ? rsqrtf(ssk + kNormEps) : 0.f;
          ms.qn[row] = (row < L) ? rsqrtf(ssq + kNormEps) : 0.f;
        }
      }
      // -- v tile -> fp16 operand (2 chunks of 8 values per thread)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int x = pt + kPrepGroupThreads * j;
        const int i = x >> 3, cc = x & 7;
        const uint4 raw = *reinterpret_cast<const uint4 *>(rv + i * kBV + 8 * cc);
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
        const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
        const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
        *reinterpret_cast<uint4 *>(sm + Lay::vh + umma::sw128_chunk(i, cc)) =
            make_uint4(pack_half2(f0.x, f0.y), pack_half2(f1.x, f1.y), pack_half2(f2.x, f2.y),
                       pack_half2(f3.x, f3.y));
      }
      // -- per-token decays alpha = 2^la2 of this thread's 16 rows (la2 from the prep kernel)
      //    and their product over the block (two channels per thread, packed f32x2 arithmetic)
      float2 al[16], bt = make_float2(1.f, 1.f), pre, suf, kts[16];
      {
        const __half *lr = reinterpret_cast<const __half *>(rg);
        const float2 one = make_float2(1.f, 1.f);
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          const int i = 16 * J + rr;
          float2 la;
          if constexpr (CPT == 2) la = __half22float2(*reinterpret_cast<const __half2 *>(lr + i * K + 2 * cg));
          else la = make_float2(__half2float(lr[i * K + cg]), 0.f);
          al[rr] = (i < L) ? make_float2(ex2_approx(la.x), ex2_approx(la.y)) : one;
          bt = __fmul2_rn(bt, al[rr]);
        }
      }
      ms.btot[J][cg * CPT] = bt.x;
      if constexpr (CPT == 2) ms.btot[J][cg * CPT + 1] = bt.y;
      umma::named_bar(kBarPrep, kPrepGroupThreads);   // norms, block products visible
      // -- decayed operands: kG = khat Gamma and q~ = qhat Gamma (forward), k~ = khat Gamma_last / Gamma
      {
        float a[2] = {1.f, 1.f}, b[2] = {1.f, 1.f};
#pragma unroll
        for (int e = 0; e < CPT; ++e) {
          const int c = cg * CPT + e;
#pragma unroll
          for (int M = 0; M < 4; ++M) {
            if (M < J) a[e] *= ms.btot[M][c];
            if (M > J) b[e] *= ms.btot[M][c];
          }
        }
        pre = make_float2(a[0], a[1]);
        suf = make_float2(b[0], b[1]);
        if (J == 0) {
          ms.gam[n & 1][cg * CPT] = a[0] * bt.x * b[0];
          if constexpr (CPT == 2) ms.gam[n & 1][cg * CPT + 1] = a[1] * bt.y * b[1];
        }
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        const int i = 16 * J + rr;
        float2 kv, qv;
        if constexpr (CPT == 2) {
          kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(rk + i * K + 2 * cg));
          qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(rq + i * K + 2 * cg));
        } else {
          kv = make_float2(__bfloat162float(rk[i * K + cg]), 0.f);
          qv = make_float2(__bfloat162float(rq[i * K + cg]), 0.f);
        }
        const float kn = ms.kn[i], qn = ms.qn[i];
        pre = __fmul2_rn(pre, al[rr]);
        const float2 kg = __fmul2_rn(kv, __fmul2_rn(pre, make_float2(kn, kn)));
        const float2 qq = __fmul2_rn(qv, __fmul2_rn(pre, make_float2(qn, qn)));
        if constexpr (CPT == 2) {
          *reinterpret_cast<uint32_t *>(sm + Lay::kG + col_panel + umma::sw128_offset(i, col_in)) =
              pack_half2(kg.x, kg.y);
          *reinterpret_cast<uint32_t *>(qt + i * K + cg * CPT) = pack_half2(qq.x, qq.y);
        } else {
          *reinterpret_cast<__half *>(sm + Lay::kG + col_panel + umma::sw128_offset(i, col_in)) =
              __float2half_rn(kg.x);
          qt[i * K + cg * CPT] = __float2half_rn(qq.x);
        }
      }
#pragma unroll
      for (int rr = 15; rr >= 0; --rr) {
        const int i = 16 * J + rr;
        float2 kv;
        if constexpr (CPT == 2) kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(rk + i * K + 2 * cg));
        else kv = make_float2(__bfloat162float(rk[i * K + cg]), 0.f);
        const float kn = ms.kn[i];
        kts[rr] = __fmul2_rn(kv, __fmul2_rn(suf, make_float2(kn, kn)));
        suf = __fmul2_rn(suf, al[rr]);
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::named_bar(kBarPrep, kPrepGroupThreads);   // kG, vh, qt complete; raw inputs consumed
      if (pt == 0) {
        wait_bar(&ms.bar_m, par);
        m_done += bad ? 0u : 1u;
      }
      if (pt == 0 && !bad) {   // D1 = M (khat Gamma), D2 = M v
        umma::fence_after_sync();
        const uint32_t id1 = umma::idesc_f16(128, K, 0, 1), id2 = umma::idesc_f16(128, kBV, 0, 1);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
          const uint64_t a = umma::sdesc_sw128(sbase + Lay::Mh + ks * 32, 16, 1024);
          umma::mma_f16_ss(tD1, a, umma::sdesc_sw128(sbase + Lay::kG + ks * 2048, Lay::kPanel64, 1024), id1,
                           ks > 0);
          umma::mma_f16_ss(tD2, a, umma::sdesc_sw128(sbase + Lay::vh + ks * 2048, Lay::kPanel64, 1024), id2,
                           ks > 0);
        }
        umma::commit(&ms.bar_d12);
      }
      if (n + 1 < nch) stage_inputs(n + 1);   // raw inputs of chunk n are consumed
      wait_bar(&ms.bar_d12, par);
      if (n + 1 < nch) stage_mats(n + 1);                 // M is consumed by D1/D2

      // -- WQ rows: w = -D1 (rows < 64), Q' = q~ - D1 (rows >= 64); WQ must be free (MMA1 of n-1 done)
      if (n > 0) wait_bar(&ms.bar_mma1, par ^ 1u);
      {
        const int row = (warp & 3) * 32 + lane;        // TMEM lane of this warp's quadrant
        const int cbeg = (warp >= 8) ? K / 2 : 0;       // warps 4-7: low half of the columns
#pragma unroll 1
        for (int c0 = cbeg; c0 < cbeg + K / 2; c0 += 16) {
          float x[16];
          umma::tmem_ld16(tD1 + lane_base + c0, x);
          umma::tmem_ld_wait();
          if (row < kChunk) {
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = -x[j];
          } else {
            const __half2 *qr = reinterpret_cast<const __half2 *>(qt + (row - kChunk) * K + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float2 f = __half22float2(qr[j]);
              x[2 * j] = f.x - x[2 * j];
              x[2 * j + 1] = f.y - x[2 * j + 1];
            }
          }
          const uint32_t pan = Lay::WQ + (uint32_t)(c0 >> 6) * (128 * 128);
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            uint4 w;
            w.x = pack_half2(x[8 * hc + 0], x[8 * hc + 1]);
            w.y = pack_half2(x[8 * hc + 2], x[8 * hc + 3]);
            w.z = pack_half2(x[8 * hc + 4], x[8 * hc + 5]);
            w.w = pack_half2(x[8 * hc + 6], x[8 * hc + 7]);
            *reinterpret_cast<uint4 *>(sm + pan + umma::sw128_chunk(row, ((c0 & 63) >> 3) + hc)) = w;
          }
        }
      }
      // -- k~ operand; it must be free (MMA2 of n-1 done)
      if (n > 0) wait_bar(&ms.bar_mma2, par ^ 1u);
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        const int i = 16 * J + rr;
        if constexpr (CPT == 2) {
          *reinterpret_cast<uint32_t *>(sm + Lay::kT + col_panel + umma::sw128_offset(i, col_in)) =
              pack_half2(kts[rr].x, kts[rr].y);
        } else {
          *reinterpret_cast<__half *>(sm + Lay::kT + col_panel + umma::sw128_offset(i, col_in)) =
              __float2half_rn(kts[rr].x);
        }
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::named_bar(kBarPrep, kPrepGroupThreads);
      if (pt == 0 && !bad) umma::mbar_arrive(&ms.bar_wq_full);
    }
  }

  // ---- exit: no bulk copy or tensor-core work of this CTA may be in flight past this point.
  // On a normal exit every copy was waited for; after a timeout, wait (bounded) for the
  // phases that were still open.
  if (tid == 0 || pt == 0) umma::commit(&ms.bar_exit);   // arrives once this thread's MMAs are done
  umma::mbar_wait_bounded(&ms.bar_exit, 0, kWaitLimit);
  if (!is_chain && *(volatile int *)&ms.err != 0) {
    // a copy issued for a chunk that was never processed may still be landing: wait for the
    // next phase of each copy barrier (returns at once if it completes, gives up otherwise)
    umma::mbar_wait_bounded(&ms.bar_in, in_done & 1u, kWaitLimit);
    if (pt == 0) umma::mbar_wait_bounded(&ms.bar_m, m_done & 1u, kWaitLimit);
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (ms.err) {
    if (tid == 0) atomicExch(p.dev_status, kDevWaitTimeout);
  } else if (is_chain && p.final_state && tid < K) {
#pragma unroll
    for (int v = 0; v < kBV; ++v) p.final_state[(((long long)s * p.H + h) * p.V + v0 + v) * K + tid] = S[v];
  }
  if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
}

template <int K>
static cudaError_t launch_recur_t(const Problem &p, const TmaMaps &maps, cudaStream_t stream) {
  const size_t smem = RecLayout<K>::bytes;
  static_assert(sizeof(RecMisc<K>) <= 4096, "misc block");
  cudaError_t e = cudaFuncSetAttribute(recur_tc_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.H * (p.V / kBV);
  recur_tc_kernel<K><<<(unsigned)grid, kRecThreads, smem, stream>>>(p, maps);
  return cudaGetLastError();
}

cudaError_t launch_recur(const Problem &p, const TmaMaps &maps, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  return p.K == 64 ? launch_recur_t<64>(p, maps, stream) : launch_recur_t<128>(p, maps, stream);
}

}  // namespace kda
