// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace skipsm {

// Device status codes (which bounded wait gave up).  0 = clean.
enum WaitSite : int {
  kSiteDecodeKFull = 1,
  kSiteDecodeVFull = 2,
  kSiteDecodeDec = 3,
  kSiteDecodeKEmpty = 4,
  kSiteDecodeVEmpty = 5,
  kSiteDecodeDrain = 6,
  kSiteInjected = 7,
  kSitePrefillQ = 16,
  kSitePrefillKFull = 17,
  kSitePrefillVFull = 18,
  kSitePrefillKEmpty = 19,
  kSitePrefillVEmpty = 20,
  kSitePrefillSFull = 21,
  kSitePrefillPFull = 22,
  kSitePrefillODone = 23,
  kSitePrefillDrain = 24,
  kSitePrefillInjected = 25,
  kSitePrefillVDec = 26,
};

struct DecodeParams {
  const __nv_bfloat16* q;  // [B][Hq][D]
  int Hq, Hkv, G, Skv, D;
  int nblk;        // key tiles of 64
  int per;         // tiles per split
  int nsplit;      // effective splits
  float scale_log2;  // softmax scale * log2(e)
  float lam_log2;    // log2(lambda), -inf when lambda == 0
  int lam_pos;       // lambda > 0
  float* ws_o;       // [B][Hq][nsplit][D] normalised split outputs
  float* ws_lse;     // [B][Hq][nsplit] split LSE in log2 units
  unsigned long long* skip_counts;  // [Hq] or null
  uint8_t* skip_mask;               // [B][Hkv][nblk] or null
  int* status;
  long long wait_cycles;
  int inject_fault;  // test hook: wait on a barrier nothing arrives at
  const uint8_t* block_mask;  // [B][Hkv][nblk] tiles to visit, or null for all
#if SKIPSM_TRACE
  // test-only instrumentation (SKIPSM_TRACE builds): %globaltimer at the start and the end
  // of every split CTA, [linear CTA index][2]
  unsigned long long* trace;
#endif
};

struct CombineParams {
  const float* ws_o;
  const float* ws_lse;
  __nv_bfloat16* o;  // [B][Hq][D]
  float* lse;        // [B][Hq] natural log, or null
  int Hq, D, nsplit;
};

cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const DecodeParams& p, int B, cudaStream_t stream);
// shared memory of one split CTA (with the block-mask tile list when p.block_mask is set)
size_t decode_smem_bytes(const DecodeParams& p);
cudaError_t launch_combine(const CombineParams& p, int B, cudaStream_t stream);

struct PrefillParams {
  int B, Hq, Hkv, G, Sq, Skv, D;
  int causal;
  int tile_q, tile_k;
  int nqt, nkt;          // vote tiles along q / key tiles
  int nblk_q;            // 256-row CTA blocks along q
  float scale_log2;
  float lam_log2;
  int lam_pos;
  int exp_mode;          // 0 exact exponentials, 1 Rowmax-PoT weights
  int qk_e4m3;           // Q and K are e4m3
  int v_e4m3;            // V is e4m3, transposed [B][Hkv][D][Skv] (needs qk_e4m3)
  float v_descale;       // multiplies the output (the caller's V quantisation scale)
  int v_after_vote;      // load V_j only once a Q tile keeps key tile j
  const uint8_t* block_mask;  // [B][Hq][nqt][nkt] pairs to visit, or null for all
  int inject_fault;      // test hook: the softmax warps wait on a barrier nothing arrives at
  __nv_bfloat16* o;      // [B][Hq][Sq][D]
  float* lse;            // [B][Hq][Sq] or null
  unsigned long long* skip_counts;
  unsigned long long* visited_counts;
  uint8_t* skip_mask;    // [B][Hq][nqt][nkt] or null
  int* status;
  long long wait_cycles;
#if SKIPSM_TRACE
  // test-only instrumentation (SKIPSM_TRACE builds): clock64 stamps of one CTA,
  // [key tile][Q tile][16] per-tile events of the softmax and MMA warps
  unsigned long long* trace;
  int trace_cta;
#endif
};

cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, const PrefillParams& p,
                           cudaStream_t stream);

int* device_status_word();  // library-global device status word

// Unique id of the CUDA context current on this thread (cuCtxGetId), or 0 when no
// context is current or the driver entry points are unavailable.  Addresses of
// the library's __device__ arrays are cached per device together with this id and
// looked up again when it changes (another context, or a device reset that
// recreated the primary context).
unsigned long long current_context_id();

// Multiprocessors of the current device (148 on B300; 148 when it cannot be queried).
int device_sm_count();

}  // namespace skipsm
