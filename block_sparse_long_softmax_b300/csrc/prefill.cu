// Skip Softmax prefill for sm_103a (tcgen05 + TMEM + TMA).
//
// Attention is computed tile by tile with an online softmax; for each
// (query tile, key tile) the tile's row maxima are compared with the running
// row maxima and the tile is skipped — no exponentials, no P.V MMA — when every
// row satisfies exp(local max - running max) < lambda ("Accelerating
// Long-Context Inference with Skip Softmax in NVIDIA TensorRT-LLM", "Skip
// Softmax Mechanism"; "NVIDIA Introduces Skip Softmax ...", "Understanding
// Skip Softmax").  The exponential work is what a skipped tile saves on
// Blackwell, where the exp units, not the tensor cores, bound attention
// ("Approximating Softmax in Pretrained LLMs ...", Abstract).
//
// CTA = 256 query rows of one (batch, query head) = two 128-row Q tiles.
//   warp 0      TMA producer of Q (once) and the K_j ring
//   warp 2      TMA producer of the V_j ring (decoupled from the K ring)
//   warp 1      TMEM allocator and MMA issuer (the warp runs converged, one
//               elected lane issues):
//                 S_x = Q_x K_j^T   (A, B from shared memory, D in TMEM)
//                 O_x += P_x V_j    (A = P from TMEM, B = V from shared memory)
//   warp 3      idle
//   warps 4-7   softmax of both Q tiles, in the order (x=0, j), (x=1, j),
//                 (x=0, j+1), ...: one thread per row = one TMEM lane; the whole
//                 S row is read into registers by one reduced load that also
//                 returns the row max (tcgen05.ld.red), the row max votes, and
//                 for kept tiles bf16 P is written over S in TMEM
// While the softmax warps work on one Q tile the tensor core runs P.V and the
// next Q.K^T of the other.  Each SMSP hosts one softmax warp: a second one would
// take the issue slots the MMA-issuing warp needs (measured: the tensor core
// slows by a third when two exp-heavy warps share the issuing warp's SMSP).
// The running max used by the vote is always the exact prefix max; the
// accumulator's reference max is only moved when the max has grown by more
// than 2^8 (lazy rescaling), which changes no result.
// With e4m3 Q, K and V the weights of P.V are quantised to e4m3 relative to the
// exact running max (the reference then follows it on every increase) and P goes
// to shared memory, one buffer per Q tile, as the A operand of an e4m3 MMA.
#include "internal.h"
#include "ptx.cuh"
#include "tmem_wide.cuh"

namespace skipsm {
namespace {

constexpr int kThreads = 256;
constexpr int kQRows = 128;        // rows of one Q tile (= MMA M)
constexpr float kRescaleLog2 = 8.f;
// e4m3 P.V: the weights enter the MMA as e4m3(2^kPShift * p), p <= 1, so the largest maps
// to 256 (inside e4m3's range) and every p >= 2^-14 keeps three mantissa bits
constexpr float kPShift = 8.f;
constexpr int kNDec = 4;   // ring of per-key-tile V decisions (V loads after the vote)

// Test-only instrumentation (built with -DSKIPSM_TRACE=1 into a separate library):
// one lane of the softmax warp of TMEM quadrant 0 and of the MMA warp stamp clock64
// at fixed points of each (key tile j, Q tile x) into p.trace[(j * 2 + x) * 16 + e].
// Events: 0 softmax entry, 1 S ready, 2 row max loaded, 3 vote decided, 4 P stored,
// 5 P arrived; 6 = 1 if the CTA kept the tile (a flag, not a time); 8 MMA warp waits
// for P, 9 P seen, 10 P.V issued, 11 next Q.K^T issued and committed.
#if SKIPSM_TRACE
#define SKIPSM_STAMP(on, j, x, e, val) \
  do { if (on) p.trace[((j) * 2 + (x)) * 16 + (e)] = (val); } while (0)
#else
#define SKIPSM_STAMP(on, j, x, e, val) do { } while (0)
#endif

// F8: 0 = bf16 Q/K/V; 1 = e4m3 Q and K, bf16 V; 2 = e4m3 Q and K and e4m3 V given
// transposed (keys innermost), with P quantised to e4m3 for the second product.
template <int D, int BK, int TQ, int NK, int NV, int F8>
struct PrefillCfg {
  static constexpr bool kV8 = F8 == 2;
  // Operand rows are cut into 128-byte swizzle atoms along D: kAtoms of them,
  // kAtomElems elements each.
  static constexpr int kQKElem = F8 ? 1 : 2;
  static constexpr int kAtoms = D * kQKElem / 128;
  static constexpr int kAtomElems = 128 / kQKElem;
  static constexpr int kQTileBytes = kQRows * D * kQKElem;
  static constexpr int kKBytes = BK * D * kQKElem;
  static constexpr int kVBytes = BK * D * (kV8 ? 1 : 2);
  static constexpr int kPBytes = kV8 ? kQRows * BK : 0;    // e4m3 P of one Q tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTileBytes;
  static constexpr int kOffV = kOffK + NK * kKBytes;
  static constexpr int kOffP = kOffV + NV * kVBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  // barriers: qfull, kfull[NK], kempty[NK], vfull[NV], vempty[NV], sfull[2],
  //           pfull[2], odone[2], final, never (failure-detection test hook)
  //           vdec[kNDec] (V loads after the vote)
  static constexpr int kNBar = 1 + 2 * NK + 2 * NV + 6 + 2 + kNDec;
  static constexpr int kOffVote = kOffBar + kNBar * 8;       // [2 x][2 parity][4 warps] int
  static constexpr int kOffDec = kOffVote + 2 * 2 * 4 * 4;   // [2] int
  static constexpr int kOffNeed = kOffDec + 2 * 4;           // [kNDec] int
  static constexpr int kOffTmem = kOffNeed + kNDec * 4;      // uint32
  static constexpr int kOffAbort = kOffTmem + 4;
  static constexpr int kBytes = kOffAbort + 16;
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns: S/P of tile x at x*BK, O of tile x at 2*BK + x*D
  static constexpr int kColS0 = 0, kColS1 = BK, kColO0 = 2 * BK, kColO1 = 2 * BK + D;
  static constexpr int kTmemUsed = 2 * BK + 2 * D;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256u : 512u;
  static constexpr uint32_t kIdescQK = F8 ? idesc_e4m3(kQRows, BK) : idesc_bf16(kQRows, BK, false, false);
  // P.V: A = P (TMEM, or e4m3 in shared memory), B = V MN-major (bf16) or V^T K-major (e4m3)
  static constexpr uint32_t kIdescPV = kV8 ? idesc_e4m3(kQRows, D) : idesc_bf16(kQRows, D, false, true);
  static constexpr float kRescale = kV8 ? 0.f : kRescaleLog2;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(!F8 || D == 128, "e4m3 Q/K: one 128-byte atom per row needs D = 128");
  static_assert(!kV8 || BK == 128, "e4m3 V: one 128-byte atom of keys per row needs BK = 128");
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms");
  static_assert(BK == 64 || BK == 128, "key tile");
  static_assert(TQ == 64 || TQ == 128, "vote rows");
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ float gapf(float tile_max, float run_max) {
  if (tile_max == -INFINITY) return -INFINITY;
  if (run_max == -INFINITY) return INFINITY;
  return tile_max - run_max;
}

// Number of key tiles visible to any query row < row_end (0 if the tile is empty).
__device__ __forceinline__ int tiles_visible(int row_begin, int row_end, const PrefillParams& p,
                                             int BK) {
  if (row_begin >= p.Sq) return 0;
  row_end = min(row_end, p.Sq);
  if (!p.causal) return p.nkt;
  const int last_key = min(p.Skv - 1, row_end - 1 + (p.Skv - p.Sq));
  return last_key / BK + 1;
}

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld<64>(uint32_t taddr, uint32_t (&r)[64]) { tmem_ld64(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ld<128>(uint32_t taddr, uint32_t (&r)[128]) { tmem_ld128(taddr, r); }

// the S row and its maximum over the tile's columns, in one load
template <int N>
__device__ __forceinline__ float tmem_ld_max(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ float tmem_ld_max<64>(uint32_t taddr, uint32_t (&r)[64]) { return tmem_ld64_max(taddr, r); }
template <>
__device__ __forceinline__ float tmem_ld_max<128>(uint32_t taddr, uint32_t (&r)[128]) { return tmem_ld128_max(taddr, r); }

template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const uint32_t (&r)[32]) { tmem_st32(taddr, r); }
template <>
__device__ __forceinline__ void tmem_st<64>(uint32_t taddr, const uint32_t (&r)[64]) { tmem_st64(taddr, r); }

// VE: V_j is loaded only once a Q tile of the CTA has voted to keep key tile j (the
// softmax posts one decision per key tile); otherwise every V_j is loaded ahead.
template <int D, int BK, int TQ, int NK, int NV, bool POT, int F8, bool BM, bool VE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using C = PrefillCfg<D, BK, TQ, NK, NV, F8>;
  constexpr bool V8 = C::kV8;
  static_assert(!(VE && POT), "the Rowmax-PoT MMA loop waits for V before the votes");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV;
  const uint32_t sP = sbase + C::kOffP;   // e4m3 P of Q tile x at sP + x * kPBytes
  const uint32_t bar0 = sbase + C::kOffBar;
  const uint32_t qfull = bar0;
  auto kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kempty = [&](int s) { return bar0 + 8u * (1 + NK + s); };
  auto vfull = [&](int s) { return bar0 + 8u * (1 + 2 * NK + s); };
  auto vempty = [&](int s) { return bar0 + 8u * (1 + 2 * NK + NV + s); };
  auto sfull = [&](int x) { return bar0 + 8u * (1 + 2 * NK + 2 * NV + x); };
  auto pfull = [&](int x) { return bar0 + 8u * (3 + 2 * NK + 2 * NV + x); };
  auto odone = [&](int x) { return bar0 + 8u * (5 + 2 * NK + 2 * NV + x); };
  const uint32_t final_bar = bar0 + 8u * (7 + 2 * NK + 2 * NV);
  const uint32_t never_bar = bar0 + 8u * (8 + 2 * NK + 2 * NV);  // nothing arrives here
  auto vdec = [&](int i) { return bar0 + 8u * (9 + 2 * NK + 2 * NV + i); };
  volatile int* sneed = reinterpret_cast<volatile int*>(smem + C::kOffNeed);
  int* svote = reinterpret_cast<int*>(smem + C::kOffVote);
  volatile int* sdec = reinterpret_cast<volatile int*>(smem + C::kOffDec);
  uint32_t* stmem = reinterpret_cast<uint32_t*>(smem + C::kOffTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  const WaitCtx wc{p.wait_cycles, p.status, abort_flag};

  // ---- work item.  All CTAs of one (batch, kv head) are adjacent, GQA siblings
  // fastest and the heaviest (last) query blocks first: the CTAs resident at any
  // time then stream the same K/V, which stays in L2 while they run.
  int id = blockIdx.x;
  const int gi = id % p.G;
  id /= p.G;
  const int qblk = p.nblk_q - 1 - id % p.nblk_q;
  id /= p.nblk_q;
  const int hkv = id % p.Hkv;
  const int b = id / p.Hkv;
  const int hq = hkv * p.G + gi;
  const int qrow0 = qblk * 2 * kQRows;
  const int n0 = tiles_visible(qrow0, qrow0 + kQRows, p, BK);
  const int n1 = tiles_visible(qrow0 + kQRows, qrow0 + 2 * kQRows, p, BK);
  const int nmax = max(n0, n1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < NK; ++s) { mbar_init(kfull(s), 1); mbar_init(kempty(s), 1); }
    for (int s = 0; s < NV; ++s) { mbar_init(vfull(s), 1); mbar_init(vempty(s), 1); }
    for (int x = 0; x < 2; ++x) {
      mbar_init(sfull(x), 1);
      mbar_init(pfull(x), 4);
      mbar_init(odone(x), 1);
    }
    mbar_init(final_bar, 1);
    mbar_init(never_bar, 1);
    for (int i = 0; i < kNDec; ++i) mbar_init(vdec(i), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(stmem), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *stmem;

  if (warp < 4) {
    if ((warp == 0 || warp == 2) && lane == 0) {
      // ============================================================ TMA
      // warp 0: Q, then the K ring; warp 2: the V ring.  The two rings advance
      // independently, so a late V tile never holds back the next K tile.
      const bool is_k = warp == 0;
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      const int NS = is_k ? NK : NV;
      const uint32_t ring = is_k ? sK : sV;
      tma_prefetch_desc(map);
      const int zk = b * p.Hkv + hkv;
      if (is_k) {
        tma_prefetch_desc(&qmap);
        const int zq = b * p.Hq + hq;
        mbar_arrive_expect_tx(qfull, 2 * C::kQTileBytes);
        // Q is read once: first out of L2, so that the kv head's K and V stay
        const uint64_t pol = l2_policy_evict_first();
        for (int x = 0; x < 2; ++x)
          for (int h = 0; h < C::kAtoms; ++h)
            tma_load_3d_hint(sQ + x * C::kQTileBytes + h * kQRows * 128, &qmap, qfull,
                             h * C::kAtomElems, qrow0 + x * kQRows, zq, pol);
      }
      // with VE the V ring holds only the kept tiles, in order: the n-th loaded V tile
      // uses stage n % NV
      const bool elide = VE && !is_k;
      int issued = 0;
      for (int j = 0; j < nmax; ++j) {
        if (elide) {
          if (!mbar_wait(vdec(j % kNDec), (j / kNDec) & 1, wc, kSitePrefillVDec)) break;
          if (!sneed[j % kNDec]) continue;
        }
        const int n = elide ? issued : j;
        const int st = n % NS;
        const uint32_t empty = is_k ? kempty(st) : vempty(st);
        const uint32_t full = is_k ? kfull(st) : vfull(st);
        if (n >= NS && !mbar_wait(empty, ((n / NS) - 1) & 1, wc,
                                  is_k ? kSitePrefillKEmpty : kSitePrefillVEmpty))
          break;
        const int bytes = is_k ? C::kKBytes : C::kVBytes;
        const int atoms = is_k ? C::kAtoms : D / 64;
        const int atom_elems = is_k ? C::kAtomElems : 64;
        mbar_arrive_expect_tx(full, bytes);
        if (V8 && !is_k) {
          // V^T: rows are the D dimensions, each one 128-byte atom of the tile's keys
          tma_load_3d(ring + st * bytes, map, full, j * BK, 0, zk);
        } else {
          for (int h = 0; h < atoms; ++h)
            tma_load_3d(ring + st * bytes + h * BK * 128, map, full, h * atom_elems, j * BK, zk);
        }
        ++issued;
      }
      if (*abort_flag) {
        // let every copy this thread started land before the CTA can exit
        const long long t0 = clock64();
        if (is_k)
          while (!mbar_try_wait(qfull, 0) && clock64() - t0 < p.wait_cycles) {}
        for (int j = max(0, issued - NS); j < issued; ++j) {
          const uint32_t full = is_k ? kfull(j % NS) : vfull(j % NS);
          while (!mbar_try_wait(full, (j / NS) & 1) && clock64() - t0 < p.wait_cycles) {}
        }
      }
    } else if (warp == 1 && nmax > 0) {
      // ============================================================ MMA
      // The whole warp runs this loop converged, so descriptors and stage indices
      // stay warp-uniform; one elected lane issues each MMA and commit.
      const uint32_t issue = elect_one();
      const int nx[2] = {n0, n1};
      const uint32_t colS[2] = {C::kColS0, C::kColS1};
      const uint32_t colO[2] = {C::kColO0, C::kColO1};
      bool first_pv[2] = {true, true};
      auto wait = [&](uint32_t bar, uint32_t parity, int site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc, site));
      };
      auto issue_s = [&](int x, int ks) {
        const uint64_t qd = sdesc_sw128(sQ + x * C::kQTileBytes, 16, 1024);
        const uint64_t kd = sdesc_sw128(sK + ks * C::kKBytes, 16, 1024);
        // each MMA covers 32 bytes of the reduction (16 bf16 or 32 e4m3 elements)
#pragma unroll
        for (int kk = 0; kk < D * C::kQKElem / 32; ++kk) {
          // advance the start address (16-byte units) within / across swizzle atoms
          const uint32_t qo = ((kk >> 2) * (kQRows * 128) + (kk & 3) * 32) >> 4;
          const uint32_t ko = ((kk >> 2) * (BK * 128) + (kk & 3) * 32) >> 4;
          if constexpr (F8 != 0)
            umma_ss_f8_w(tmem + colS[x], qd + qo, kd + ko, C::kIdescQK, kk > 0 ? 1u : 0u, issue);
          else
            umma_ss_w(tmem + colS[x], qd + qo, kd + ko, C::kIdescQK, kk > 0 ? 1u : 0u, issue);
        }
      };
      auto issue_pv = [&](int x, int vs) {
        if constexpr (V8) {
          // A = e4m3 P of Q tile x (one 128-byte atom of keys per row), B = V^T (one atom of
          // keys per D row); each MMA covers 32 keys
          const uint64_t pd = sdesc_sw128(sP + x * C::kPBytes, 16, 1024);
          const uint64_t vd = sdesc_sw128(sV + vs * C::kVBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            umma_ss_f8_w(tmem + colO[x], pd + kk * 2, vd + kk * 2, C::kIdescPV,
                         (first_pv[x] && kk == 0) ? 0u : 1u, issue);
        } else {
          const uint64_t vd = sdesc_sw128(sV + vs * C::kVBytes, BK * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_ts_w(tmem + colO[x], tmem + colS[x] + kk * 8, vd + ((kk * 16 * 128) >> 4),
                      C::kIdescPV, (first_pv[x] && kk == 0) ? 0u : 1u, issue);
        }
        first_pv[x] = false;
      };
      bool ok = wait(qfull, 0, kSitePrefillQ) && wait(kfull(0), 0, kSitePrefillKFull);
      if (ok) {
        tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if (nx[x] > 0) {
            issue_s(x, 0);
            umma_commit_w(sfull(x), issue);
          }
        umma_commit_w(kempty(0), issue);
      }
#if SKIPSM_TRACE
      const bool tr_on = p.trace && static_cast<int>(blockIdx.x) == p.trace_cta && lane == 0;
#else
      const bool tr_on = false;
#endif
      (void)tr_on;
      int nv = 0;  // with VE: V tiles consumed (only kept tiles are loaded)
      for (int j = 0; ok && j < nmax; ++j) {
        const int vn = VE ? nv : j;   // the producer's count of V tiles before this one
        const int vs = vn % NV, ks1 = (j + 1) % NK;
        const uint32_t vpar = (vn / NV) & 1;
        const bool has_next = j + 1 < nmax;
        bool v_ready = false, k_ready = false;
        if constexpr (POT) {
          // V_j and K_{j+1} are needed in this iteration whatever the votes.  With the
          // longer Rowmax-PoT softmax, waiting for them before the first P (rather than
          // between that P and its MMAs) measured 3-4 % faster on the 128K prefill; with
          // exact exponentials it measured 1 % slower at lambda = 0, so the exact kernel
          // waits for each where it first uses it.
          if (!wait(vfull(vs), vpar, kSitePrefillVFull)) { ok = false; break; }
          v_ready = true;
          if (has_next) {
            if (!wait(kfull(ks1), ((j + 1) / NK) & 1, kSitePrefillKFull)) { ok = false; break; }
            k_ready = true;
          }
          tc_fence_after();
        }
        for (int x = 0; x < 2 && ok; ++x) {
          if (j >= nx[x]) continue;
          SKIPSM_STAMP(tr_on, j, x, 8, clock64());
          if (!wait(pfull(x), j & 1, kSitePrefillPFull)) { ok = false; break; }
          tc_fence_after();
          SKIPSM_STAMP(tr_on, j, x, 9, clock64());
          if (sdec[x]) {
            if (!v_ready) {
              if (!wait(vfull(vs), vpar, kSitePrefillVFull)) { ok = false; break; }
              v_ready = true;
              tc_fence_after();
            }
            issue_pv(x, vs);
          }
          SKIPSM_STAMP(tr_on, j, x, 10, clock64());
          if (j + 1 < nx[x]) {
            if (!k_ready) {  // K_{j+1} is first needed here, after P.V of tile j is queued
              if (!wait(kfull(ks1), ((j + 1) / NK) & 1, kSitePrefillKFull)) { ok = false; break; }
              k_ready = true;
              tc_fence_after();
            }
            issue_s(x, ks1);
            umma_commit_w(sfull(x), issue);
            SKIPSM_STAMP(tr_on, j, x, 11, clock64());
          } else {
            // the last tile of this Q tile: one commit lets the epilogue wait for its final P.V
            umma_commit_w(odone(x), issue);
          }
        }
        if (!ok) break;
        if (has_next) umma_commit_w(kempty(ks1), issue);
        if constexpr (VE) {
          // V_j was loaded iff some Q tile kept tile j
          if (v_ready) {
            umma_commit_w(vempty(vs), issue);
            ++nv;
          }
        } else {
          if (!v_ready && !wait(vfull(vs), vpar, kSitePrefillVFull)) break;
          umma_commit_w(vempty(vs), issue);
        }
      }
      // every MMA issued by this warp completes before TMEM is released
      umma_commit_w(final_bar, issue);
      const long long t0 = clock64();
      while (!mbar_try_wait(final_bar, 0) && clock64() - t0 < p.wait_cycles) {}
    }
  } else {
    // ============================================================ softmax
    // One warpgroup serves both Q tiles in the order the MMA warp issues them:
    // (x=0, j), (x=1, j), (x=0, j+1), ...  While it works on one tile, the tensor
    // core runs P.V and the next Q.K^T of the other, and each SMSP hosts a single
    // softmax warp, which leaves issue slots for the MMA-issuing thread.
    const int wq = warp & 3;              // TMEM lane quadrant
    const int r = wq * 32 + lane;         // row within a Q tile
    const int qoff = p.Skv - p.Sq;
    const int grp = TQ == 128 ? 0 : (wq >> 1);  // vote group within a Q tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = p.scale_log2;
    struct TileRow {
      int n, n_grp, n_half0, n_half1, qtile, row, qpos;
      int j_mask;  // first key tile in which a row of this warp has a masked key
      bool valid;
      float M, R, l;   // running max, reference max of the accumulator, row sum
    };
    TileRow tr[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int t0 = qrow0 + x * kQRows;
      const int grp_row0 = t0 + grp * TQ;
      tr[x].n = x == 0 ? n0 : n1;
      tr[x].n_grp = tiles_visible(grp_row0, grp_row0 + TQ, p, BK);
      tr[x].n_half0 = tiles_visible(t0, t0 + 64, p, BK);
      tr[x].n_half1 = tiles_visible(t0 + 64, t0 + 128, p, BK);
      tr[x].qtile = grp_row0 / TQ;
      tr[x].row = t0 + r;
      tr[x].valid = tr[x].row < p.Sq;
      tr[x].qpos = tr[x].row + qoff;
      // key tile j holds a key that is masked for some row of this warp iff its
      // last key is past the warp's smallest position (causal) or past Skv
      const int qpos_warp0 = t0 + wq * 32 + qoff;
      tr[x].j_mask = p.Skv / BK;
      if (p.causal) tr[x].j_mask = min(tr[x].j_mask, (qpos_warp0 + 1) / BK);
      tr[x].M = -INFINITY;
      tr[x].R = -INFINITY;
      tr[x].l = 0.f;
    }
    unsigned long long n_skip = 0, n_visit = 0;
    int v_posted = -1;   // (thread 0, VE) the last key tile whose V decision is posted
    bool ok = true;
    if (p.inject_fault) {
      // failure-detection test hook: a wait on a barrier nothing arrives at, with half
      // the normal bound so that it is the wait reported; the CTA then winds down
      const WaitCtx half{p.wait_cycles / 2, p.status, abort_flag};
      ok = mbar_wait(never_bar, 0, half, kSitePrefillInjected);
    }
#if SKIPSM_TRACE
    const bool tr_on = p.trace && static_cast<int>(blockIdx.x) == p.trace_cta && r == 0;
#else
    const bool tr_on = false;
#endif
    (void)tr_on;
    // e4m3 P row of Q tile x into shared memory: eight 16-byte chunks of 16 keys,
    // XOR-swizzled within the row's 128-byte atom (the MMA's 128-byte-swizzle layout).
    // P_x(j) is free to overwrite: its S was committed after the P.V that read P_x(j-1).
    auto store_p8 = [&](int x, const uint32_t (&pk)[BK / 2]) {
      const uint32_t row = sP + x * C::kPBytes + static_cast<uint32_t>(r) * 128u;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(row + ((c ^ (r & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      fence_proxy_async_smem();
    };
    bool next_ready = false;  // the S of the next tile in this order is known to be complete
    // The softmax of one (Q tile x, key tile j): t is the row state of Q tile x, o that of the
    // other Q tile.
    auto softmax_tile = [&](TileRow& t, const TileRow& o, const int x, const int j) {
      if (j >= t.n) return;
      // caller's block mask: a (vote tile, key tile) pair outside it is not visited
      bool sel0 = true, sel1 = true;  // vote groups 0 and 1 of this Q tile
      if constexpr (BM) {
        const int qt0 = (qrow0 + x * kQRows) / TQ;
        const uint8_t* mcol = p.block_mask + (static_cast<size_t>(b) * p.Hq + hq) * p.nqt * p.nkt + j;
        sel0 = mcol[static_cast<size_t>(qt0) * p.nkt] != 0;
        sel1 = TQ == 128 ? sel0 : (qt0 + 1 < p.nqt && mcol[static_cast<size_t>(qt0 + 1) * p.nkt] != 0);
      }
      const uint32_t tS = lane_base + (x == 0 ? C::kColS0 : C::kColS1);
      const uint32_t tO = lane_base + (x == 0 ? C::kColO0 : C::kColO1);
      SKIPSM_STAMP(tr_on, j, x, 0, clock64());
      if (!next_ready) ok = mbar_wait(sfull(x), j & 1, wc, kSitePrefillSFull) && ok;
      tc_fence_after();
      SKIPSM_STAMP(tr_on, j, x, 1, clock64());
      uint32_t sv[BK];
      // the load also returns the row's maximum over the tile (tcgen05.ld.red)
      float mx = tmem_ld_max<BK>(tS, sv);
      SKIPSM_STAMP(tr_on, j, x, 2, clock64());
      const int key0 = j * BK;
      // tile-level (warp-uniform) test: does any row of this warp see a masked key?
      if (j >= t.j_mask) {
#pragma unroll
        for (int i = 0; i < BK; ++i) {
          const int key = key0 + i;
          const bool masked = (p.causal && key > t.qpos) || key >= p.Skv;
          sv[i] = masked ? __float_as_uint(-INFINITY) : sv[i];
        }
        // the maximum over the visible keys: 16 independent chains, then a tree
        float m16[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) m16[k] = __uint_as_float(sv[k]);
#pragma unroll
        for (int i = 16; i < BK; i += 16)
#pragma unroll
          for (int k = 0; k < 16; ++k) m16[k] = fmaxf(m16[k], __uint_as_float(sv[i + k]));
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int k = 0; k < w; ++k) m16[k] = fmaxf(m16[k], m16[k + w]);
        mx = m16[0];
      }
      const float mt2 = t.valid ? mx * sl2 : -INFINITY;
      const float d = gapf(mt2, t.M);
      const bool row_vote = !t.valid || d < p.lam_log2;
      bool skip_g[2];
      if (TQ == 128) {
        // one vote group = the whole Q tile: a barrier that ANDs the row votes
        // (every warp does exactly one barrier operation per tile, so the warps
        // stay matched even when a bounded wait has given up)
        bool sk;
        if constexpr (BM)  // an unselected tile is the same for every warp: no barrier
          sk = !sel0 || (p.lam_pos && named_bar_and(1 + x, 128, row_vote));
        else
          sk = p.lam_pos && named_bar_and(1 + x, 128, row_vote);
        skip_g[0] = skip_g[1] = sk;
      } else {
      const bool warp_vote = __all_sync(0xffffffffu, row_vote);
      volatile int* vote = svote + (x * 2 + (j & 1)) * 4;
      if (lane == 0) vote[wq] = warp_vote ? 1 : 0;
      // A warp with a row that keeps the tile knows its vote group keeps it, so it
      // only arrives on the barrier; warps whose rows all vote skip wait for every
      // vote.  A 64-row group past its causal range never keeps the tile.  Every
      // warp does exactly one barrier operation per tile, so the warps stay
      // matched even when a bounded wait has given up.
      bool out_of_range = j >= (grp == 0 ? t.n_half0 : t.n_half1);
      if constexpr (BM) out_of_range = out_of_range || !(grp == 0 ? sel0 : sel1);
      if ((!warp_vote || !p.lam_pos) && !out_of_range) {
        named_bar_arrive(1 + x, 128);
        // this group keeps the tile; the other group's decision is not needed (written
        // with selects: an index by the warp's group would put skip_g in local memory)
        skip_g[0] = grp != 0;
        skip_g[1] = grp == 0;
      } else {
        named_bar_sync(1 + x, 128);
        const int v0 = vote[0], v1 = vote[1], v2 = vote[2], v3 = vote[3];
        // tiles past a 64-row group's causal range, or outside the block mask, are
        // not visited by it
        skip_g[0] = (p.lam_pos && (v0 & v1 & 1)) || j >= t.n_half0;
        skip_g[1] = (p.lam_pos && (v2 & v3 & 1)) || j >= t.n_half1;
        if constexpr (BM) {
          skip_g[0] = skip_g[0] || !sel0;
          skip_g[1] = skip_g[1] || !sel1;
        }
      }
      }
      const bool any_kept = !(skip_g[0] && skip_g[1]);
      const bool my_skip = grp == 0 ? skip_g[0] : skip_g[1];
      SKIPSM_STAMP(tr_on, j, x, 3, clock64());
      SKIPSM_STAMP(tr_on, j, x, 6, any_kept ? 1ull : 0ull);
      bool counted = r == grp * TQ && j < t.n_grp;  // one thread per vote group records it
      if constexpr (BM) counted = counted && (grp == 0 ? sel0 : sel1);
      if (counted) {
        ++n_visit;
        n_skip += my_skip ? 1 : 0;
        if (p.skip_mask)
          p.skip_mask[((static_cast<size_t>(b) * p.Hq + hq) * p.nqt + t.qtile) * p.nkt + j] =
              my_skip ? 1 : 0;
      }
      if (r == 0) {
        sdec[x] = any_kept ? 1 : 0;
        if constexpr (VE) {
          // V_j is fetched once some Q tile keeps tile j: at the first Q tile that keeps it,
          // or at the last Q tile that visits it
          const bool last_visit = x == 1 || j >= n1;
          if (v_posted != j && (any_kept || last_visit)) {
            sneed[j % kNDec] = any_kept ? 1 : 0;
            mbar_arrive(vdec(j % kNDec));
            v_posted = j;
          }
        }
      }
      if (any_kept) {
        if (!my_skip) {
          t.M = fmaxf(t.M, mt2);
          float alpha = 1.f;
          bool resc = false;
          if (t.M > t.R + C::kRescale) {   // also true for the first kept tile (R = -inf)
            resc = t.R != -INFINITY;
            alpha = ex2(t.R - t.M);
            t.l *= alpha;
            t.R = t.M;
          }
          if (__any_sync(0xffffffffu, resc)) {
            // Every earlier P.V of this Q tile is complete: the S of this tile was
            // committed after it, and the next P.V waits for this warpgroup.

            // 32 columns at a time: the S row is still live in registers
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t ov[32];
              tmem_ld32(tO + c0, ov);
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tmem_st32(tO + c0, ov);
            }
          }
          float la[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[BK / 2];
          if constexpr (V8) {
            // P = 2^(s*scale*log2e - M + 8) rounded to e4m3 (the 2^8 cancels in O / l),
            // written to shared memory in the 128-byte-swizzle layout of a K-major operand
            float negR = kPShift - t.R;
            if constexpr (BM) negR = t.R == -INFINITY ? 0.f : negR;
#pragma unroll
            for (int i = 0; i < BK / 4; ++i) {
              float x0, x1, x2, x3;
              ffma2(x0, x1, __uint_as_float(sv[4 * i]), __uint_as_float(sv[4 * i + 1]), sl2, negR);
              ffma2(x2, x3, __uint_as_float(sv[4 * i + 2]), __uint_as_float(sv[4 * i + 3]), sl2, negR);
              const float e0 = ex2(x0), e1 = ex2(x1), e2 = ex2(x2), e3 = ex2(x3);
              fadd2_acc(la[0], la[1], e0, e1);
              fadd2_acc(la[2], la[3], e2, e3);
              pk[i] = pack_e4m3x4(e0, e1, e2, e3);
            }
          } else if constexpr (!POT) {
            // P = 2^(s*scale*log2e - R) in bf16, written over S (a row that has
            // seen no key yet, R = -inf, only has masked keys here: P = 0)
            float negR = -t.R;
            if constexpr (BM) negR = t.R == -INFINITY ? 0.f : negR;
#pragma unroll
            for (int i = 0; i < BK / 2; ++i) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]), sl2, negR);
              const float e0 = ex2(x0), e1 = ex2(x1);
              fadd2_acc(la[2 * (i & 1)], la[2 * (i & 1) + 1], e0, e1);
              pk[i] = pack_bf16x2(e0, e1);
            }
          } else {
            // Rowmax-PoT ("Approximating Softmax in Pretrained LLMs ...", Abstract):
            // the weight is 2^n, n = round(x), x = s*scale*log2e - M, anchored at the
            // running row max M, and 0 below 2^-126.5.  One saturating FMA gives
            // u = clamp(1 + x/127, 0, 1) (masked keys, -inf, give 0); adding
            // 1.5*2^23 - 127 to 127*u rounds x to n (ties to even) and leaves the fp32
            // bits 0x4B400000 + n; shifting those bits by 23 and adding the bits of
            // 1.0 builds the fp32 bits of 2^n (n = -127 gives 0).  The factor
            // 2^(M - R) to the accumulator's reference R is rounded to bf16, so
            // P = 2^n * c is exact in bf16 and the row sum adds exactly what the MMA
            // multiplies.  The fp32 error of x is below 3e-5, well inside the band
            // in which the exponent's rounding is treated as ambiguous.
            const float ua = sl2 * (1.f / 127.f);
            const float ub = 1.f - t.M * (1.f / 127.f);
            float c = __bfloat162float(__float2bfloat16_rn(ex2(t.M - t.R)));
            if constexpr (BM) c = t.R == -INFINITY ? 0.f : c;
#pragma unroll
            for (int i = 0; i < BK / 2; ++i) {
              const float u0 = sat_fma(__uint_as_float(sv[2 * i]), ua, ub);
              const float u1 = sat_fma(__uint_as_float(sv[2 * i + 1]), ua, ub);
              float y0, y1;
              ffma2(y0, y1, u0, u1, 127.f, 12582912.f - 127.f);
              const float p0 = __uint_as_float(__float_as_uint(y0) * 8388608u + 0x3F800000u);
              const float p1 = __uint_as_float(__float_as_uint(y1) * 8388608u + 0x3F800000u);
              float e0, e1;
              ffma2(e0, e1, p0, p1, c, 0.f);
              fadd2_acc(la[2 * (i & 1)], la[2 * (i & 1) + 1], e0, e1);
              pk[i] = pack_bf16x2(e0, e1);
            }
          }
          t.l += (la[0] + la[1]) + (la[2] + la[3]);
          if constexpr (V8) {
            store_p8(x, pk);
          } else {
            tmem_st<BK / 2>(tS, pk);
          }
        } else {
          uint32_t z[BK / 2];
#pragma unroll
          for (int i = 0; i < BK / 2; ++i) z[i] = 0u;
          if constexpr (V8) {
            store_p8(x, z);
          } else {
            tmem_st<BK / 2>(tS, z);
          }
        }
      }
      SKIPSM_STAMP(tr_on, j, x, 4, clock64());
      {
        // Probe the next tile's S without blocking; its latency overlaps the
        // fence and arrive below, and a complete phase skips the wait.
        int xn = 1 - x, jn = x == 0 ? j : j + 1, nn = o.n;
        if (jn >= nn) { xn = x; jn = j + 1; nn = t.n; }
        next_ready = jn < nn && mbar_test_wait(sfull(xn), jn & 1);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull(x));
      SKIPSM_STAMP(tr_on, j, x, 5, clock64());
    };
    if constexpr (POT) {
      // One copy of the longer Rowmax-PoT body serves both Q tiles (x at run time, the row
      // states swapping places): held once in the instruction caches it measured 17 % faster
      // than two copies with a constant x, which the exact and FP8 bodies prefer (4-9 %).
      TileRow ta = tr[0], tb = tr[1];
#pragma unroll 1
      for (int hs = 0; hs < 2 * nmax; ++hs) {
        if (hs > 0) {
          const TileRow tmp = ta;
          ta = tb;
          tb = tmp;
        }
        softmax_tile(ta, tb, hs & 1, hs >> 1);
      }
      if (nmax > 0) {  // the last half-step was Q tile 1
        tr[0] = tb;
        tr[1] = ta;
      }
    } else {
      for (int j = 0; j < nmax; ++j) {
        softmax_tile(tr[0], tr[1], 0, j);
        softmax_tile(tr[1], tr[0], 1, j);
      }
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      TileRow& t = tr[x];
      if (__all_sync(0xffffffffu, ok && t.n > 0 && !*abort_flag)) {  // warp-uniform: TMEM loads below
        // ---- epilogue: O / l -> bf16, LSE (one commit after the last P.V of this Q tile)
        ok = mbar_wait(odone(x), 0, wc, kSitePrefillODone);
        tc_fence_after();
        uint32_t ov[D];
        tmem_ld<D>(lane_base + (x == 0 ? C::kColO0 : C::kColO1), ov);
        if (t.valid && ok) {
          float inv = 1.f / t.l;
          __nv_bfloat16* orow = p.o + ((static_cast<size_t>(b) * p.Hq + hq) * p.Sq + t.row) * D;
          uint4* dst = reinterpret_cast<uint4*>(orow);
          // (e4m3 P.V: l carries the 2^8 of the weights, and O the caller's V scale)
          float lse2 = t.R + __log2f(t.l) - (V8 ? kPShift : 0.f);
          if constexpr (V8) inv *= p.v_descale;
          if constexpr (BM) {
            // a row with no visited visible key (block mask) has l = 0: output 0, LSE -inf
            if (!(t.l > 0.f)) {
#pragma unroll
              for (int i = 0; i < D; ++i) ov[i] = 0u;
              inv = 0.f;
              lse2 = -INFINITY;
            }
          }
          const uint64_t opol = l2_policy_evict_first();   // O is written once
#pragma unroll
          for (int i = 0; i < D / 8; ++i)
            st_global_v4_hint(dst + i, make_uint4(
                pack_bf16x2(__uint_as_float(ov[8 * i]) * inv, __uint_as_float(ov[8 * i + 1]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv, __uint_as_float(ov[8 * i + 3]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv, __uint_as_float(ov[8 * i + 5]) * inv),
                pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv, __uint_as_float(ov[8 * i + 7]) * inv)), opol);
          if (p.lse)
            p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Sq + t.row] = lse2 * 0.69314718055994531f;
        }
      }
    }
    if (r == grp * TQ) {
      if (p.skip_counts && n_skip) atomicAdd(p.skip_counts + hq, n_skip);
      if (p.visited_counts && n_visit) atomicAdd(p.visited_counts + hq, n_visit);
    }
  }

  // ---- teardown: TMEM is freed only after every MMA and TMEM access is done
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int BK, int TQ, int NK, int NV, bool POT, int F8, bool BM, bool VE = false>
cudaError_t launch_cfg(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       const PrefillParams& p, cudaStream_t stream) {
  using C = PrefillCfg<D, BK, TQ, NK, NV, F8>;
  auto kern = prefill_kernel<D, BK, TQ, NK, NV, POT, F8, BM, VE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kAlloc);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(p.nblk_q) * p.B * p.Hq;
  kern<<<grid, kThreads, C::kAlloc, stream>>>(qmap, kmap, vmap, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, const PrefillParams& p, cudaStream_t stream) {
  // template flags: Rowmax-PoT weights, e4m3 Q/K, caller block mask
#define SKIPSM_PREFILL_FLAGS(d, bk, tq, nk, nv, f8)                                           \
  {                                                                                         \
    const bool pot = p.exp_mode == 1, bm = p.block_mask != nullptr;                         \
    if (pot && bm) return launch_cfg<d, bk, tq, nk, nv, true, f8, true>(qmap, kmap, vmap, p, stream);   \
    if (pot) return launch_cfg<d, bk, tq, nk, nv, true, f8, false>(qmap, kmap, vmap, p, stream);        \
    if (bm) return launch_cfg<d, bk, tq, nk, nv, false, f8, true>(qmap, kmap, vmap, p, stream);         \
    return launch_cfg<d, bk, tq, nk, nv, false, f8, false>(qmap, kmap, vmap, p, stream);                \
  }
#define SKIPSM_PREFILL_CASE(d, bk, tq, nk, nv)                                 \
  if (p.D == d && p.tile_k == bk && p.tile_q == tq && !p.qk_e4m3)          \
    SKIPSM_PREFILL_FLAGS(d, bk, tq, nk, nv, 0)
  // V loads after the vote (bf16, D = 128, 128-key tiles, exact exponentials)
  if (p.v_after_vote && p.D == 128 && p.tile_k == 128 && !p.qk_e4m3 && p.exp_mode == 0) {
    const bool bm = p.block_mask != nullptr;
    if (p.tile_q == 128)
      return bm ? launch_cfg<128, 128, 128, 3, 2, false, 0, true, true>(qmap, kmap, vmap, p, stream)
                : launch_cfg<128, 128, 128, 3, 2, false, 0, false, true>(qmap, kmap, vmap, p, stream);
    return bm ? launch_cfg<128, 128, 64, 3, 2, false, 0, true, true>(qmap, kmap, vmap, p, stream)
              : launch_cfg<128, 128, 64, 3, 2, false, 0, false, true>(qmap, kmap, vmap, p, stream);
  }
  SKIPSM_PREFILL_CASE(128, 128, 128, 3, 2)
  SKIPSM_PREFILL_CASE(128, 128, 64, 3, 2)
  SKIPSM_PREFILL_CASE(128, 64, 128, 4, 4)
  SKIPSM_PREFILL_CASE(128, 64, 64, 4, 4)
  SKIPSM_PREFILL_CASE(64, 128, 128, 4, 3)
  SKIPSM_PREFILL_CASE(64, 128, 64, 4, 3)
  SKIPSM_PREFILL_CASE(64, 64, 128, 6, 6)
  SKIPSM_PREFILL_CASE(64, 64, 64, 6, 6)
  // e4m3 Q and K: 128-row vote groups or 64, 128-key tiles, D = 128
  if (p.qk_e4m3 && !p.v_e4m3 && p.D == 128 && p.tile_k == 128) {
    if (p.tile_q == 128) SKIPSM_PREFILL_FLAGS(128, 128, 128, 4, 3, 1)
    SKIPSM_PREFILL_FLAGS(128, 128, 64, 4, 3, 1)
  }
  // e4m3 Q, K and V (exact exponentials quantised to e4m3 for P.V)
  if (p.qk_e4m3 && p.v_e4m3 && p.D == 128 && p.tile_k == 128 && p.exp_mode == 0) {
    const bool bm = p.block_mask != nullptr;
    if (p.tile_q == 128)
      return bm ? launch_cfg<128, 128, 128, 4, 3, false, 2, true>(qmap, kmap, vmap, p, stream)
                : launch_cfg<128, 128, 128, 4, 3, false, 2, false>(qmap, kmap, vmap, p, stream);
    return bm ? launch_cfg<128, 128, 64, 4, 3, false, 2, true>(qmap, kmap, vmap, p, stream)
              : launch_cfg<128, 128, 64, 4, 3, false, 2, false>(qmap, kmap, vmap, p, stream);
  }
#undef SKIPSM_PREFILL_CASE
#undef SKIPSM_PREFILL_FLAGS
  return cudaErrorInvalidValue;
}

}  // namespace skipsm
