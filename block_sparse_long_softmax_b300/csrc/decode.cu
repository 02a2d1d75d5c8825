// Skip Softmax decode for sm_103a: split-KV GQA attention of one query token
// per sequence, with the block-skip rule of "Accelerating Long-Context
// Inference with Skip Softmax in NVIDIA TensorRT-LLM" ("Skip Softmax
// Mechanism"): a 64-key tile is skipped when, for every query head of the GQA
// group, exp(local max - running max) < lambda.  A skipped tile's V rows are
// never fetched — the memory-bandwidth saving the pages describe for decoding
// ("NVIDIA Introduces Skip Softmax ...", "Benefits and Implementation").
//
// One CTA = one (split, kv head, batch).  Warp 4 is the TMA producer: it keeps
// NK key tiles in flight and fetches a value tile only after the consumers'
// vote on it.  Warps 0-3 each own 16 keys of every tile:
//   S-phase (tile i):   S^T[16 keys x 8 heads] = K Q^T   (mma.sync m16n8k16)
//                       per-head tile max -> vote -> exp -> P^T fragments
//   PV-phase (tile i-LAG): O^T[D x 8 heads] += V^T P^T   (if tile kept)
// so the V load of a kept tile overlaps LAG tiles of key streaming.  The
// split result (O / l, log2 LSE) goes to the workspace; a second kernel merges
// the splits with an exact log-sum-exp combine.
//
// With a caller-supplied block mask ("NVIDIA Introduces Skip Softmax ...",
// "Benefits and Implementation": Skip Softmax combined with a block selector)
// the CTA first compacts the selected tiles of its split into a list in shared
// memory; every role then walks that list instead of the whole split, so an
// unselected tile is never read.
#include "internal.h"
#include "ptx.cuh"

namespace skipsm {
namespace {

constexpr int kBk = 64;             // keys per tile
constexpr int kConsumers = 128;     // 4 warps
constexpr int kThreads = 160;       // + 1 producer warp
constexpr int kNDec = 8;            // decision ring (>= NK)

template <int D, int NK, int NV, int LAG>
struct DecodeCfg {
  static constexpr int kStageBytes = kBk * D * 2;  // 8 KB (D=64) / 16 KB (D=128)
  static constexpr int kNSlot = LAG + 1;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + NK * kStageBytes;
  static constexpr int kOffSlot = kOffV + NV * kStageBytes;
  static constexpr int kSlotBytes = 4 * 32 * 32;  // per tile: 4 warps x 32 lanes x (float4, uint2 P, pad)
  static constexpr int kOffRed = kOffSlot + kNSlot * kSlotBytes;      // [2][4][8] float
  static_assert(kOffSlot % 16 == 0, "slot entries hold float4");
  static constexpr int kOffLRed = kOffRed + 2 * 4 * 8 * 4;            // [4][8] float
  static constexpr int kOffRRed = kOffLRed + 4 * 8 * 4;               // [8] float
  static constexpr int kOffAb = kOffRRed + 8 * 4;                     // [3][4] int abort votes
  static constexpr int kOffDec = kOffAb + 3 * 4 * 4;                  // [kNDec] int
  static constexpr int kOffBar = kOffDec + kNDec * 4;                 // mbarriers (8 B each)
  static constexpr int kNBar = 2 * NK + 2 * NV + kNDec + 1;
  static constexpr int kOffAbort = kOffBar + kNBar * 8;
  static constexpr int kBytes = kOffAbort + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  // block-mask tile list: [count int, pad to 16][uint16 tile offsets within the split]
  static constexpr int kOffSel = (kBytes + 15) & ~15;
  static_assert(4 * D * 8 * 4 <= NK * kStageBytes, "final reduction buffer aliases K stages");
  static_assert(NK <= kNDec, "decision ring must cover the key prefetch depth");
};

__device__ __forceinline__ float gap(float tile_max, float run_max) {
  // tile max - running max, +inf before any key (never happens for a valid
  // head after its first tile), -inf for an empty row
  if (tile_max == -INFINITY) return -INFINITY;
  if (run_max == -INFINITY) return INFINITY;
  return tile_max - run_max;
}

template <int D, int NK, int NV, int LAG>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using C = DecodeCfg<D, NK, NV, LAG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t kst = sbase + C::kOffK, vst = sbase + C::kOffV;
  float* sred = reinterpret_cast<float*>(smem + C::kOffRed);
  float* lred = reinterpret_cast<float*>(smem + C::kOffLRed);
  float* rred = reinterpret_cast<float*>(smem + C::kOffRRed);
  int* sdec = reinterpret_cast<int*>(smem + C::kOffDec);
  volatile int* sab = reinterpret_cast<volatile int*>(smem + C::kOffAb);  // [parity/final][warp]
  const uint32_t bar0 = sbase + C::kOffBar;
  auto kfull = [&](int i) { return bar0 + 8u * i; };
  auto kempty = [&](int i) { return bar0 + 8u * (NK + i); };
  auto vfull = [&](int i) { return bar0 + 8u * (2 * NK + i); };
  auto vempty = [&](int i) { return bar0 + 8u * (2 * NK + NV + i); };
  auto decbar = [&](int i) { return bar0 + 8u * (2 * NK + 2 * NV + i); };
  const uint32_t never_bar = bar0 + 8u * (2 * NK + 2 * NV + kNDec);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);

  // Launch order: split-major, the last split of every (batch, kv head) first.  The last
  // split holds the most recent keys, where the most tiles are kept, so the heaviest CTAs
  // start in the first wave and the lightest (first splits) fill the tail.
  const int lin = blockIdx.x + p.nsplit * (blockIdx.y + p.Hkv * blockIdx.z);
  const int ngroups = p.Hkv * static_cast<int>(gridDim.z);
  const int grp_id = lin % ngroups;
  const int split = p.nsplit - 1 - lin / ngroups, hkv = grp_id % p.Hkv, b = grp_id / p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#if SKIPSM_TRACE
  const size_t cta_lin = (static_cast<size_t>(b) * p.Hkv + hkv) * p.nsplit + split;
  if (p.trace && threadIdx.x == 0) p.trace[2 * cta_lin] = globaltimer_ns();
#endif
  const int j0 = split * p.per;
  const int nb = min(p.per, p.nblk - j0);
  const WaitCtx wc{p.wait_cycles, p.status, abort_flag};

  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) { mbar_init(kfull(i), 1); mbar_init(kempty(i), 4); }
    for (int i = 0; i < NV; ++i) { mbar_init(vfull(i), 1); mbar_init(vempty(i), 4); }
    for (int i = 0; i < kNDec; ++i) mbar_init(decbar(i), 1);
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  int* snsel = reinterpret_cast<int*>(smem + C::kOffSel);
  uint16_t* sel = reinterpret_cast<uint16_t*>(smem + C::kOffSel + 16);
  if (p.block_mask && warp == 0) {
    // compact the selected tiles of this split (ascending) with ballots
    const uint8_t* mrow = p.block_mask + (static_cast<size_t>(b) * p.Hkv + hkv) * p.nblk + j0;
    int cnt = 0;
    for (int base = 0; base < nb; base += 32) {
      const int i = base + lane;
      const bool on = i < nb && mrow[i] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, on);
      if (on) sel[cnt + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(i);
      cnt += __popc(bal);
    }
    if (lane == 0) *snsel = cnt;
  }
  __syncthreads();
  // tiles this CTA visits, and the split-relative index of the i-th of them
  const int nvis = p.block_mask ? *snsel : nb;
  auto tile_of = [&](int i) { return p.block_mask ? static_cast<int>(sel[i]) : i; };

  // ------------------------------------------------------------ producer --
  if (warp == 4) {
    if (lane != 0) return;
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    const int zc = b * p.Hkv + hkv;
    int k_issued[NK];
    int v_issued[NV];
#pragma unroll
    for (int i = 0; i < NK; ++i) k_issued[i] = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) v_issued[i] = 0;
    auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int tile) {
      mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
      for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * 8192, map, bar, h * 64, tile * kBk, zc);
    };
    for (int s = 0; s < NK && s < nvis; ++s) {
      load_tile(&kmap, kst + s * C::kStageBytes, kfull(s), j0 + tile_of(s));
      k_issued[s] = 1;
    }
    int nv = 0;
    for (int i = 0; i < nvis; ++i) {
      if (!mbar_wait(decbar(i % kNDec), (i / kNDec) & 1, wc, kSiteDecodeDec)) break;
      if (sdec[i % kNDec]) {
        const int vs = nv % NV;
        if (nv >= NV && !mbar_wait(vempty(vs), ((nv / NV) - 1) & 1, wc, kSiteDecodeVEmpty)) break;
        load_tile(&vmap, vst + vs * C::kStageBytes, vfull(vs), j0 + tile_of(i));
        ++v_issued[vs];
        ++nv;
      }
      if (i + NK < nvis) {
        const int ks = i % NK;
        if (!mbar_wait(kempty(ks), (i / NK) & 1, wc, kSiteDecodeKEmpty)) break;
        load_tile(&kmap, kst + ks * C::kStageBytes, kfull(ks), j0 + tile_of(i + NK));
        ++k_issued[ks];
      }
    }
    if (*abort_flag) {
      // let every copy this CTA started land before the CTA can exit
      const long long t0 = clock64();
#pragma unroll
      for (int s = 0; s < NK; ++s)
        if (k_issued[s])
          while (!mbar_try_wait(kfull(s), (k_issued[s] - 1) & 1) && clock64() - t0 < p.wait_cycles) {}
#pragma unroll
      for (int s = 0; s < NV; ++s)
        if (v_issued[s])
          while (!mbar_try_wait(vfull(s), (v_issued[s] - 1) & 1) && clock64() - t0 < p.wait_cycles) {}
    }
    return;
  }

  // ----------------------------------------------------------- consumers --
  const int g = lane >> 2, t = lane & 3;
  const int hA = 2 * t, hB = 2 * t + 1;
  const int G = p.G;

  if (p.inject_fault && threadIdx.x == 0) {
    // half the normal bound, so this wait (the injected root cause) is the one reported
    const WaitCtx half{p.wait_cycles / 2, p.status, abort_flag};
    mbar_wait(never_bar, 0, half, kSiteInjected);
  }
  __syncwarp();

  uint32_t qf[D / 16][2];
  {
    const __nv_bfloat16* qg = p.q + (static_cast<size_t>(b) * p.Hq + hkv * G) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      if (g < G) {
        qf[kk][0] = *reinterpret_cast<const uint32_t*>(qg + g * D + 16 * kk + 2 * t);
        qf[kk][1] = *reinterpret_cast<const uint32_t*>(qg + g * D + 16 * kk + 8 + 2 * t);
      } else {
        qf[kk][0] = qf[kk][1] = 0u;
      }
    }
  }

  float MA = -INFINITY, MB = -INFINITY;  // running max (log2 units)
  float RA = -INFINITY, RB = -INFINITY;  // max the accumulator is scaled to
  float lA = 0.f, lB = 0.f;
  float o[D / 16][4];
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  uint32_t kept_hist = 0;
  int n_pv = 0, n_skip = 0;
  const float sl2 = p.scale_log2;
  uint8_t* slot_base = smem + C::kOffSlot;

  for (int i = 0; i < nvis + LAG; ++i) {
    if (i < nvis) {
      // ---- S-phase of tile i
      const int st = i % NK;
      mbar_wait(kfull(st), (i / NK) & 1, wc, kSiteDecodeKFull);
      __syncwarp();  // the spin-wait may leave lanes diverged; ldmatrix/mma need the full warp
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t kb = kst + st * C::kStageBytes;
      const int krow = 16 * warp + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int chunk = 2 * kk + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kb + (chunk >> 3) * 8192 + swz128(krow, chunk & 7), a0, a1, a2, a3);
        mma_bf16_16816(acc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(kempty(st));
      const int jt = j0 + tile_of(i);  // key tile index
      const int key0 = jt * kBk + 16 * warp + g;
      const float s0 = key0 < p.Skv ? acc[0] * sl2 : -INFINITY;
      const float s1 = key0 < p.Skv ? acc[1] * sl2 : -INFINITY;
      const float s2 = key0 + 8 < p.Skv ? acc[2] * sl2 : -INFINITY;
      const float s3 = key0 + 8 < p.Skv ? acc[3] * sl2 : -INFINITY;
      float mA = fmaxf(s0, s2), mB = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(0xffffffffu, mA, off));
        mB = fmaxf(mB, __shfl_xor_sync(0xffffffffu, mB, off));
      }
      float* red = sred + (i & 1) * 32;
      if (lane < 4) { red[warp * 8 + 2 * lane] = mA; red[warp * 8 + 2 * lane + 1] = mB; }
      if (lane == 0) sab[(i & 1) * 4 + warp] = *abort_flag;
      named_bar_sync(1, kConsumers);
      // every consumer warp takes the same decision from the four recorded flags
      if (sab[(i & 1) * 4] | sab[(i & 1) * 4 + 1] | sab[(i & 1) * 4 + 2] | sab[(i & 1) * 4 + 3]) break;
      const float tA = fmaxf(fmaxf(red[hA], red[8 + hA]), fmaxf(red[16 + hA], red[24 + hA]));
      const float tB = fmaxf(fmaxf(red[hB], red[8 + hB]), fmaxf(red[16 + hB], red[24 + hB]));
      const float dA = gap(tA, MA), dB = gap(tB, MB);
      const bool vote = (hA >= G || dA < p.lam_log2) && (hB >= G || dB < p.lam_log2);
      const bool skip = __all_sync(0xffffffffu, vote) && p.lam_pos;
      MA = fmaxf(MA, tA);
      MB = fmaxf(MB, tB);
      if (threadIdx.x == 0) {
        sdec[i % kNDec] = skip ? 0 : 1;
        mbar_arrive(decbar(i % kNDec));
        if (p.skip_mask)
          p.skip_mask[(static_cast<size_t>(b) * p.Hkv + hkv) * p.nblk + jt] = skip ? 1 : 0;
      }
      n_skip += skip ? 1 : 0;
      kept_hist = (kept_hist << 1) | (skip ? 0u : 1u);
      __syncwarp();
      if (!skip) {
        const float p0 = ex2(s0 - MA), p1 = ex2(s1 - MB), p2 = ex2(s2 - MA), p3 = ex2(s3 - MB);
        uint8_t* slot = slot_base + (i % C::kNSlot) * C::kSlotBytes + (warp * 32 + lane) * 32;
        *reinterpret_cast<float4*>(slot) = make_float4(MA, MB, p0 + p2, p1 + p3);
        *reinterpret_cast<uint2*>(slot + 16) =
            make_uint2(movmatrix_t(pack_bf16x2(p0, p1)), movmatrix_t(pack_bf16x2(p2, p3)));
      }
    } else {
      kept_hist <<= 1;
    }
    // ---- PV-phase of tile i - LAG
    if (i >= LAG && ((kept_hist >> LAG) & 1u)) {
      const int vs = n_pv % NV;
      mbar_wait(vfull(vs), (n_pv / NV) & 1, wc, kSiteDecodeVFull);
      __syncwarp();
      const uint8_t* slot =
          slot_base + ((i - LAG) % C::kNSlot) * C::kSlotBytes + (warp * 32 + lane) * 32;
      const float4 mf = *reinterpret_cast<const float4*>(slot);
      const uint2 pf = *reinterpret_cast<const uint2*>(slot + 16);
      const float aA = ex2(RA - mf.x), aB = ex2(RB - mf.y);
      RA = mf.x;
      RB = mf.y;
      lA = lA * aA + mf.z;
      lB = lB * aB + mf.w;
      const uint32_t vb = vst + vs * C::kStageBytes;
      const int vrow = 16 * warp + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[mt][0] *= aA; o[mt][1] *= aB; o[mt][2] *= aA; o[mt][3] *= aB;
        const int chunk = 2 * mt + ((lane >> 3) & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vb + (chunk >> 3) * 8192 + swz128(vrow, chunk & 7), a0, a1, a2, a3);
        mma_bf16_16816(o[mt], a0, a1, a2, a3, pf.x, pf.y);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(vempty(vs));
      ++n_pv;
    }
  }

  // ---- merge the four warps' partial results (reuses the K stages)
  if (lane == 0) sab[8 + warp] = *abort_flag;
  named_bar_sync(1, kConsumers);
  if (sab[8] | sab[9] | sab[10] | sab[11]) return;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }
  float* ored = reinterpret_cast<float*>(smem + C::kOffK);  // [4][D][8]
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    float* ow = ored + (warp * D + 16 * mt + g) * 8;
    ow[hA] = o[mt][0];
    ow[hB] = o[mt][1];
    ow[64 + hA] = o[mt][2];  // dim + 8
    ow[64 + hB] = o[mt][3];
  }
  if (g == 0) {
    lred[warp * 8 + hA] = lA;
    lred[warp * 8 + hB] = lB;
    if (warp == 0) { rred[hA] = RA; rred[hB] = RB; }
  }
  named_bar_sync(1, kConsumers);
  const size_t row0 = static_cast<size_t>(b) * p.Hq + hkv * G;
  for (int idx = threadIdx.x; idx < G * D; idx += kConsumers) {
    const int h = idx / D, d = idx % D;
    const float sum = ored[(0 * D + d) * 8 + h] + ored[(1 * D + d) * 8 + h] +
                      ored[(2 * D + d) * 8 + h] + ored[(3 * D + d) * 8 + h];
    const float l = lred[h] + lred[8 + h] + lred[16 + h] + lred[24 + h];
    p.ws_o[((row0 + h) * p.nsplit + split) * D + d] = l > 0.f ? sum / l : 0.f;
  }
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    const float l = lred[h] + lred[8 + h] + lred[16 + h] + lred[24 + h];
    // a split with no visited tile (block mask) weighs nothing in the combine
    p.ws_lse[(row0 + h) * p.nsplit + split] = l > 0.f ? rred[h] + __log2f(l) : -INFINITY;
  }
  if (threadIdx.x == 0 && p.skip_counts && n_skip) {
    for (int h = 0; h < G; ++h)
      atomicAdd(p.skip_counts + hkv * G + h, static_cast<unsigned long long>(n_skip));
  }
#if SKIPSM_TRACE
  if (p.trace && threadIdx.x == 0) p.trace[2 * cta_lin + 1] = globaltimer_ns();
#endif
}

// One CTA per (b, query head); thread d merges dimension d over the splits.
__global__ void decode_combine_kernel(const CombineParams p) {
  const int row = blockIdx.x;  // b * Hq + h
  const float* lse = p.ws_lse + static_cast<size_t>(row) * p.nsplit;
  float top = -INFINITY;
  for (int s = 0; s < p.nsplit; ++s) top = fmaxf(top, lse[s]);
  if (top == -INFINITY) {  // no visited key at all (block mask): output 0, LSE -inf
    for (int d = threadIdx.x; d < p.D; d += blockDim.x)
      p.o[static_cast<size_t>(row) * p.D + d] = __float2bfloat16_rn(0.f);
    if (p.lse && threadIdx.x == 0) p.lse[row] = -INFINITY;
    return;
  }
  float wsum = 0.f;
  for (int s = 0; s < p.nsplit; ++s) wsum += ex2(lse[s] - top);
  for (int d = threadIdx.x; d < p.D; d += blockDim.x) {
    float acc = 0.f;
    const float* os = p.ws_o + static_cast<size_t>(row) * p.nsplit * p.D + d;
    for (int s = 0; s < p.nsplit; ++s) acc += ex2(lse[s] - top) * os[static_cast<size_t>(s) * p.D];
    p.o[static_cast<size_t>(row) * p.D + d] = __float2bfloat16_rn(acc / wsum);
  }
  if (p.lse && threadIdx.x == 0) p.lse[row] = (top + __log2f(wsum)) * 0.69314718055994531f;
}

template <int D, int NK, int NV, int LAG>
size_t split_smem(const DecodeParams& p) {
  using C = DecodeCfg<D, NK, NV, LAG>;
  // the list region starts at most 15 bytes past kBytes: pad by 16
  return p.block_mask ? C::kAlloc + 16 + ((2 * static_cast<size_t>(p.per) + 15) & ~size_t(15)) + 16
                      : C::kAlloc;
}

template <int D, int NK, int NV, int LAG>
cudaError_t launch_split(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                         int B, cudaStream_t stream) {
  auto kern = decode_split_kernel<D, NK, NV, LAG>;
  const size_t smem = split_smem<D, NK, NV, LAG>(p);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.nsplit, p.Hkv, B);
  kern<<<grid, kThreads, smem, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

// The default split count assumes two split CTAs resident per SM (228 KB of shared memory
// per SM, 1 KB of it reserved per CTA); both configurations below must keep that.
static_assert(2 * (DecodeCfg<128, 3, 2, 2>::kAlloc + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(2 * (DecodeCfg<64, 6, 3, 2>::kAlloc + 1024) <= 228 * 1024, "two CTAs per SM");

}  // namespace

size_t decode_smem_bytes(const DecodeParams& p) {
  return p.D == 128 ? split_smem<128, 3, 2, 2>(p) : split_smem<64, 6, 3, 2>(p);
}

// P.V runs two tiles behind the vote (LAG = 2), so a kept tile's value fetch, which can only
// start once the tile is voted on, has two tiles of key streaming to land in.  D = 128 keeps
// three key tiles in flight: against four key tiles and LAG = 1 this measured 4-8 % faster at
// skip ratios 0.24-0.81 and no slower at lambda = 0 (128K: 613 against 618 us).  D = 64 keeps
// six: against LAG = 1, 3-6 % faster at every measured skip ratio (128K: 399 against 423 us at
// lambda = 0).
cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                          int B, cudaStream_t stream) {
  if (p.D == 128) return launch_split<128, 3, 2, 2>(kmap, vmap, p, B, stream);
  return launch_split<64, 6, 3, 2>(kmap, vmap, p, B, stream);
}

cudaError_t launch_combine(const CombineParams& p, int B, cudaStream_t stream) {
  decode_combine_kernel<<<B * p.Hq, p.D, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace skipsm
