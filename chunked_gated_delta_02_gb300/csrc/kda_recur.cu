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
// The prep kernel hands over M, khat Gamma and k~ (as swizzled operand images),
// q~ and Gamma_last per chunk; v comes straight from the input by TMA. D1 and D2 are
// one product M [khat Gamma | v], and WQ is written to tensor memory, where MMA1
// reads its A operand: shared-memory bandwidth, which every tcgen05.mma operand
// and every staged copy shares, bounds this kernel.
//
// Warp roles (the S-independent work of chunk n+1 overlaps the state chain of
// chunk n):
//   chain group, warps 0-3: D2 += WQ S, U and o, D3 = k~^T U, S update.
//   prep group, warps 4-11: stages the chunk's operands (bulk copies and one
//     TMA tile of v), converts v to fp16, issues D1 and D2, and forms WQ.
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
  // two input buffers (chunk parity), each [M (128 x 64 K-major, A of D12) | khat Gamma | v (fp16)]:
  // khat Gamma (64 x K) and v (64 x 64) are consecutive MN-major panels, the B operand of
  // D12 = M [khat Gamma | v]
  static constexpr uint32_t mk = 0;
  static constexpr uint32_t mk_kg = 128 * 128, mk_vh = mk_kg + (K / 64) * kPanel64, mk_size = mk_vh + kPanel64;
  static constexpr uint32_t Sh = mk + 2 * mk_size;               // K x 64    MN-major (B of MMA1)
  static constexpr uint32_t Uh = Sh + K * 128;                   // 64 x 64   MN-major (B of MMA2)
  static constexpr uint32_t rv = Uh + kPanel64;                  // 2 x bf16 v [64][64]
  // two chunk buffers, each [k~ (64 x 128 MN-major, A of MMA2) | q~ image (64 x K) | Gamma_last (K fp32)]
  static constexpr uint32_t qb = rv + 2 * 64 * kBV * 2;
  static constexpr uint32_t qb_kt = 0, qb_qt = 2 * kPanel64, qb_gam = qb_qt + 128 * K;
  static constexpr uint32_t qb_size = (qb_gam + 4 * K + 1023) / 1024 * 1024;
  static constexpr uint32_t misc = qb + 2 * qb_size;
  static constexpr uint32_t bytes = misc + 1024 + 1024;          // + misc + alignment slack
};

// Tensor memory columns: D12 = [D1 | D2] of chunk parity b at b (K + 64) (D2 accumulates the
// chain's WQ S), D3 after both, then WQ (fp16 pairs, the A operand of MMA1).
template <int K>
struct RecTmem {
  static constexpr uint32_t d12 = K + 64;
  static constexpr uint32_t d3 = 2 * d12, wq = d3 + 64;
  static_assert(wq + K / 2 <= 512, "tensor memory columns");
};

// Small per-CTA state after the operand buffers.
struct RecMisc {
  uint64_t bar_d12, bar_wq_full, bar_mma1, bar_mma2[2], bar_exit, bar_in[2], bar_q;
  uint32_t tmem_slot;
  int err;
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

template <int K>
__global__ void __launch_bounds__(kRecThreads, 1)
recur_tc_kernel(const Problem p, const __grid_constant__ TmaMaps maps) {
  using Lay = RecLayout<K>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so that the
  // compiler keeps every access in the shared address space
  unsigned char *sm = smem_raw + ((1024u - (umma::smem_u32(smem_raw) & 1023u)) & 1023u);
  RecMisc &ms = *reinterpret_cast<RecMisc *>(sm + Lay::misc);

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

  // ---- set-up: zero the k~ operands (rows >= K stay zero when K = 64), TMEM, barriers
  for (int b = 0; b < 2; ++b)
    for (int x = tid; x < (int)(2 * Lay::kPanel64 / 16); x += kRecThreads)
      reinterpret_cast<uint4 *>(sm + Lay::qb + b * Lay::qb_size + Lay::qb_kt)[x] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    umma::tmem_alloc(&ms.tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    umma::mbar_init(&ms.bar_d12, 1);
    umma::mbar_init(&ms.bar_wq_full, 1);
    umma::mbar_init(&ms.bar_mma1, 1);
    umma::mbar_init(&ms.bar_mma2[0], 1);   // D3 of even / odd chunks
    umma::mbar_init(&ms.bar_mma2[1], 1);
    umma::mbar_init(&ms.bar_exit, 2);
    umma::mbar_init(&ms.bar_in[0], 1);
    umma::mbar_init(&ms.bar_in[1], 1);
    umma::mbar_init(&ms.bar_q, 1);
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
  // Operands of chunk n (hand-off block of its (chunk, head) slot), in two groups:
  //   bar_in[n & 1]: [M | khat Gamma] (one bulk copy) and the v tile (64 x 64 at column v0, one
  //           TMA copy; tokens past T read as zeros, tokens of the next packed sequence are zeroed
  //           after arrival) into input buffer n & 1; consumed by D1 / D2. Issued by prep thread 0.
  //   bar_q:  [k~ | q~ | Gamma_last] into chunk buffer n & 1 (one bulk copy when K = 128); k~ is
  //           consumed by D3, q~ by the WQ rows, Gamma_last by the state update. Issued by prep
  //           thread 32, so that its cost is off the path of thread 0.
  auto stage_in = [&](int n) {
    if (pt == 0) {
      const unsigned char *hb = p.hand + (((long long)si.chunk0 + n) * p.H + h) * p.hand_stride;
      uint64_t *bar = &ms.bar_in[n & 1];
      static_assert(Lay::mk_kg == hand_off_kg(K), "input buffer layout");
      umma::mbar_arrive_expect_tx(bar, (uint32_t)(hand_off_kt(K) + kChunk * kBV * 2));
      umma::bulk_g2s(sm + Lay::mk + (n & 1) * Lay::mk_size, hb, (uint32_t)hand_off_kt(K), bar);
      umma::tma_load_4d(sm + Lay::rv + (n & 1) * (kChunk * kBV * 2), &maps.v, v0, h, si.t0 + n * kChunk, si.b, bar);
    }
  };
  auto stage_q = [&](int n) {
    if (pt == 32) {
      const unsigned char *hb = p.hand + (((long long)si.chunk0 + n) * p.H + h) * p.hand_stride;
      unsigned char *qb = sm + Lay::qb + (n & 1) * Lay::qb_size;
      umma::mbar_arrive_expect_tx(&ms.bar_q, 2 * kChunk * K * 2 + K * 4);
      if constexpr (K == 128) {   // the smem buffer has the global block's internal offsets
        static_assert(Lay::qb_qt == hand_off_qt(K) - hand_off_kt(K) && Lay::qb_gam == hand_off_gam(K) - hand_off_kt(K),
                      "chunk buffer layout");
        umma::bulk_g2s(qb, hb + hand_off_kt(K), (uint32_t)(hand_off_gam(K) + 4 * K - hand_off_kt(K)), &ms.bar_q);
      } else {
        umma::bulk_g2s(qb + Lay::qb_kt, hb + hand_off_kt(K), kChunk * K * 2, &ms.bar_q);
        umma::bulk_g2s(qb + Lay::qb_qt, hb + hand_off_qt(K), kChunk * K * 2, &ms.bar_q);
        umma::bulk_g2s(qb + Lay::qb_gam, hb + hand_off_gam(K), K * 4, &ms.bar_q);
      }
    }
  };
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  if (!is_chain && nch > 0) {
    stage_in(0);
    stage_q(0);
  }
  const uint32_t tmem = ms.tmem_slot;
  using Tm = RecTmem<K>;
  const uint32_t tD3 = tmem + Tm::d3, tWQ = tmem + Tm::wq;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  bool bad = false;   // this thread saw a wait time out
  uint32_t in_done0 = 0, in_done1 = 0, q_done = 0;   // completed bar_in[0], bar_in[1], bar_q phases seen

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
      const uint32_t tD2 = tmem + Tm::d12 * (n & 1) + K;
      const int t0 = si.t0 + n * kChunk;
      const int L = min(kChunk, si.len - n * kChunk);
      wait_bar(&ms.bar_wq_full, par);
      const float gam = (tid < K) ? reinterpret_cast<const float *>(sm + Lay::qb + (n & 1) * Lay::qb_size +
                                                                     Lay::qb_gam)[tid]
                                  : 0.f;   // read before MMA1: the buffer is reused
      if (tid == 0 && !bad) {   // D2 += WQ S  ->  [-U ; O]
        const uint32_t id = umma::idesc_f16(128, kBV, 0, 1);
        const uint64_t b0 = umma::sdesc_sw128(sbase + Lay::Sh, K * 128, 1024);
#pragma unroll
        for (int ks = 0; ks < K / 16; ++ks) umma::mma_f16_ts(tD2, tWQ + ks * 8, umma::desc_add(b0, ks * 2048), id, 1);
        umma::commit(&ms.bar_mma1);
      }
      wait_bar(&ms.bar_mma1, par);
      // U (rows < 64) -> fp16 operand; o = scale * O (rows >= 64) -> bf16 global
#pragma unroll 1
      for (int c0 = 0; c0 < kBV; c0 += 32) {
        float x[32];
        umma::tmem_ld32(tD2 + lane_base + c0, x);
        umma::tmem_ld_wait();
        if (tid < kChunk) {
#pragma unroll
          for (int hc = 0; hc < 4; ++hc) {
            uint4 w;
            w.x = pack_half2(-x[8 * hc + 0], -x[8 * hc + 1]);
            w.y = pack_half2(-x[8 * hc + 2], -x[8 * hc + 3]);
            w.z = pack_half2(-x[8 * hc + 4], -x[8 * hc + 5]);
            w.w = pack_half2(-x[8 * hc + 6], -x[8 * hc + 7]);
            *reinterpret_cast<uint4 *>(sm + Lay::Uh + umma::sw128_chunk(tid, (c0 >> 3) + hc)) = w;
          }
        } else if (tid - kChunk < L && !bad) {
          uint4 *dst = reinterpret_cast<uint4 *>(p.o + tok_row(p, si.b, t0 + tid - kChunk, h) * p.V + v0 + c0);
#pragma unroll
          for (int hc = 0; hc < 4; ++hc) {
            __nv_bfloat16 ob[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) ob[j] = __float2bfloat16_rn(p.scale * x[8 * hc + j]);
            dst[hc] = *reinterpret_cast<const uint4 *>(ob);
          }
        }
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      umma::named_bar(kBarChain, kChainThreads);
      if (tid == 0 && !bad) {   // D3 = k~^T U
        umma::fence_after_sync();
        const uint32_t id = umma::idesc_f16(128, kBV, 1, 1);
        const uint64_t a0 =
            umma::sdesc_sw128(sbase + Lay::qb + (n & 1) * Lay::qb_size + Lay::qb_kt, Lay::kPanel64, 1024);
        const uint64_t b0 = umma::sdesc_sw128(sbase + Lay::Uh, Lay::kPanel64, 1024);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)
          umma::mma_f16_ss(tD3, umma::desc_add(a0, ks * 2048), umma::desc_add(b0, ks * 2048), id, ks > 0);
        umma::commit(&ms.bar_mma2[n & 1]);
      }
      wait_bar(&ms.bar_mma2[n & 1], (uint32_t)((n >> 1) & 1));
      // S = gamma S + D3 (thread = channel), fp16 copy for the next chunk
      if (tid < K) {
#pragma unroll
        for (int c0 = 0; c0 < kBV; c0 += 32) {
          float x[32];
          umma::tmem_ld32(tD3 + lane_base + c0, x);
          umma::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) S[c0 + j] = fmaf(gam, S[c0 + j], x[j]);
#pragma unroll
          for (int hc = 0; hc < 4; ++hc) {
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
    // Software-pipelined one chunk ahead: after releasing chunk n to the chain, the group
    // converts v of chunk n + 1 and issues its D1 / D2, so that they run during the chain's
    // work on chunk n.
    // Input buffer m & 1 of chunk m: wait for its copies, zero the v rows past the sequence end,
    // convert v to fp16, then issue D1 = M (khat Gamma) and D2 = M v (commit on bar_d12).
    auto start_chunk = [&](int m) {
      const int b = m & 1;
      const int L = min(kChunk, si.len - m * kChunk);
      __nv_bfloat16 *rvb = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::rv + b * (kChunk * kBV * 2));
      wait_bar(&ms.bar_in[b], (uint32_t)((m >> 1) & 1));
      if (!bad) {
        if (b) ++in_done1;
        else ++in_done0;
      }
      if (L < kChunk) {   // v rows past the sequence end (next packed sequence or zero fill): zero them
        for (int x = pt; x < (kChunk - L) * (kBV / 8); x += kPrepGroupThreads) {
          const int i = L + x / (kBV / 8), c8 = x % (kBV / 8);
          *reinterpret_cast<uint4 *>(rvb + i * kBV + 8 * c8) = make_uint4(0, 0, 0, 0);
        }
        umma::named_bar(kBarPrep, kPrepGroupThreads);
      }
      const uint32_t mkb = Lay::mk + b * Lay::mk_size;
      // v tile -> fp16 operand, the panel after khat Gamma (2 chunks of 8 values per thread)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int x = pt + kPrepGroupThreads * j;
        const int i = x >> 3, cc = x & 7;
        const uint4 raw = *reinterpret_cast<const uint4 *>(rvb + i * kBV + 8 * cc);
        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
        const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
        const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
        *reinterpret_cast<uint4 *>(sm + mkb + Lay::mk_vh + umma::sw128_chunk(i, cc)) =
            make_uint4(pack_half2(f0.x, f0.y), pack_half2(f1.x, f1.y), pack_half2(f2.x, f2.y),
                       pack_half2(f3.x, f3.y));
      }
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      // vh complete, the v tile consumed; also the group's agreement to stop after an error
      const bool stop = umma::bar_red_or(kBarPrep, kPrepGroupThreads, bad || *(volatile int *)&ms.err != 0);
      if (pt == 0 && !stop) {   // D12 = M [khat Gamma | v] = [[-w ; P w] | [-u ; P u]]
        umma::fence_after_sync();
        const uint32_t id = umma::idesc_f16(128, K + kBV, 0, 1);
        const uint64_t a0 = umma::sdesc_sw128(sbase + mkb, 16, 1024);
        const uint64_t b0 = umma::sdesc_sw128(sbase + mkb + Lay::mk_kg, Lay::kPanel64, 1024);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks)
          umma::mma_f16_ss(tmem + Tm::d12 * b, umma::desc_add(a0, ks * 32), umma::desc_add(b0, ks * 2048), id, ks > 0);
        umma::commit(&ms.bar_d12);
      }
      return stop;
    };
    if (nch > 1) stage_in(1);
    bool stop = (nch > 0) ? start_chunk(0) : false;
    for (int n = 0; n < nch; ++n) {
      const uint32_t par = (uint32_t)(n & 1);
      if (stop) break;   // uniform over the group (decided by a barrier reduction)
      wait_bar(&ms.bar_d12, par);         // D1 / D2 of chunk n are done
      if (n + 2 < nch) stage_in(n + 2);   // ... so input buffer n & 1 is free
      wait_bar(&ms.bar_q, par);
      q_done += bad ? 0u : 1u;

      // -- WQ rows: w = -D1 (rows < 64), Q' = q~ - D1 (rows >= 64), as fp16 pairs into tensor memory;
      //    WQ must be free (MMA1 of n-1 done)
      if (n > 0) wait_bar(&ms.bar_mma1, par ^ 1u);
      {
        const uint32_t tD1 = tmem + Tm::d12 * (n & 1);
        const int row = (warp & 3) * 32 + lane;        // TMEM lane of this warp's quadrant
        const int cbeg = (warp >= 8) ? K / 2 : 0;       // warps 4-7: low half of the columns
#pragma unroll 1
        for (int c0 = cbeg; c0 < cbeg + K / 2; c0 += 32) {
          float x[32];
          umma::tmem_ld32(tD1 + lane_base + c0, x);
          umma::tmem_ld_wait();
          if (row < kChunk) {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = -x[j];
          } else {   // q~ row (row - 64), columns c0 .. c0 + 31: four swizzled 16-byte chunks
            const int qi = row - kChunk;
            const unsigned char *qrow = sm + Lay::qb + (n & 1) * Lay::qb_size + Lay::qb_qt +
                                        (uint32_t)(c0 >> 6) * Lay::kPanel64 + (uint32_t)qi * 128;
#pragma unroll
            for (int hc = 0; hc < 4; ++hc) {
              const uint4 raw = *reinterpret_cast<const uint4 *>(qrow + (((((c0 & 63) >> 3) + hc) ^ (qi & 7)) << 4));
              const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(h2[e]);
                x[8 * hc + 2 * e] = f.x - x[8 * hc + 2 * e];
                x[8 * hc + 2 * e + 1] = f.y - x[8 * hc + 2 * e + 1];
              }
            }
          }
#pragma unroll
          for (int hs = 0; hs < 2; ++hs) {
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) pk[j] = pack_half2(x[16 * hs + 2 * j], x[16 * hs + 2 * j + 1]);
            umma::tmem_st8(tWQ + lane_base + (uint32_t)((c0 + 16 * hs) >> 1), pk);
          }
        }
        umma::tmem_st_wait();
      }
      umma::fence_proxy_async_smem();   // q~ reads before the bulk copy that later reuses the buffer
      umma::fence_before_sync();
      umma::named_bar(kBarPrep, kPrepGroupThreads);   // WQ complete
      if (pt == 0 && !bad) umma::mbar_arrive(&ms.bar_wq_full);
      // Chunk buffer (n + 1) & 1 was last read by D3 and the state update of chunk n - 1 (and its
      // q~ by the WQ rows of chunk n - 1), and D2 of chunk n + 1 overwrites the accumulator that
      // the chain read for chunk n - 1: wait for D3 of chunk n - 1. Its barrier only carries the
      // products of odd or of even chunks, and the next phase (chunk n + 1) cannot complete
      // before chunk n + 1 is released, so the wait cannot mistake one phase for another.
      if (n > 0) wait_bar(&ms.bar_mma2[(n - 1) & 1], (uint32_t)(((n - 1) >> 1) & 1));
      if (n + 1 < nch && !bad) stage_q(n + 1);
      if (n + 1 < nch) stop = start_chunk(n + 1);
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
    // input buffer b has seen in_done[b] phases; a copy may be open for its next one
    umma::mbar_wait_bounded(&ms.bar_in[0], in_done0 & 1u, kWaitLimit);
    umma::mbar_wait_bounded(&ms.bar_in[1], in_done1 & 1u, kWaitLimit);
    umma::mbar_wait_bounded(&ms.bar_q, q_done & 1u, kWaitLimit);
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
  static_assert(sizeof(RecMisc) <= 1024, "misc block");
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
