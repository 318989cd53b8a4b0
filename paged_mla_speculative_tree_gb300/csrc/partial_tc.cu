// Tensor-core (tcgen05 / TMEM) split-K partial kernel for MLA tree-verify
// attention on sm_103a.
//
// Work unit: a pair of CTAs (a 2-CTA cluster) owns 128 query rows of one
// request -- two draft-tree tokens x 64 heads -- and one split of the
// request's keys (prefix keys through kv_indices, then the tree tokens through
// out_cache_loc: "The Final Solder Joint" -- "The Three-Edits Sequence").
// Each latent row gathered from the paged pool is shared by all 64 heads x
// both tokens of the tile ("The Glue That Connects" -- "The Context": the
// MLA latent is read once instead of once per head).
//
// The 576 contraction dims are split between the two CTAs: CTA c holds latent
// dims [256c, 256c+256) and rope dims [32c, 32c+32).  Per 64-key tile:
//   1. two gather warps copy the CTA's 576 bytes of each latent row with
//      cp.async (16 B per lane, one row per warp instruction) into a
//      128B-swizzled K-major tile (64B swizzle for the rope part); invalid
//      slots are zero-filled; each lane's copies complete on the stage's
//      barrier, so the warps never wait for memory.  (Scattered 1152-byte
//      rows: per-warp cp.async scales with the number of issuing warps, while
//      TMA gathers are limited to about one 128-byte row per 18 cycles per SM);
//   2. GEMM1 on the tensor core: S_c[128 x 64] = Q_c . K_c^T, fp32 in TMEM;
//      the latent part of Q_c is the A operand in TMEM (16 k-steps), its rope
//      part an A operand in shared memory (2 k-steps);
//   3. the softmax warps (one per TMEM lane quarter by default, all 64 key
//      columns of its 32 rows) send their partial S to the peer CTA: each
//      warp stages its 32 rows in shared memory and issues one bulk copy that
//      completes bytes on the peer's barrier (double-buffered, one tile
//      ahead).  The values travel as 16-bit integers relative to the midpoint
//      of each row's NCOL values, with a power-of-two step per row: the error
//      of a partial score is at most 2^-15 (1 + 2^-10) of the row's half-range
//      (max - min)/2, whatever the size of the scores (the distributed-shared-
//      memory link, ~17 B/cycle per CTA, is what this exchange costs, which
//      rules out fp32).  Then the warps add the peer's partial to their own
//      exact one, apply the tree mask (prefix always visible, tree columns
//      from custom_mask), and run the fp32 online softmax ("Design Decisions
//      and Trade-Offs": mask -> -inf, streaming max/sum) with a lazily moved
//      reference max; P (bf16) goes to one of two TMEM buffers.  Each CTA
//      normalises its own O half with its own softmax sums (of the weights
//      rounded to bf16, as GEMM2 uses them), so the two views of S need not
//      be bit-identical;
//   4. GEMM2: O_c[128 x 256] += P (TMEM, A operand) . V_c, where V_c is this
//      CTA's 256 latent dims of the same smem tile read as an MN-major operand.
// The end of a split writes the normalised partial O halves and the LSE of
// CTA 0 (or the final bf16 output when there is one split).
//
// TMEM (512 columns): O half [0,256), partial S [256,320), latent Q half
// [320,448), P double buffer [448,512).
//
// Every pipeline wait is bounded (Params::wait_cycles).  A wait that gives up
// sets MTV_DEVERR_TIMEOUT and the abort flag of both CTAs of the pair, and
// every role leaves its loop.  The wind-down then runs with its own bound and
// ignores the abort flag: the MMA issuer waits for a final commit (every MMA
// it issued has completed), the gather warps wait for their copies, each
// softmax warp tells the peer how many score tiles it sent, and after a
// cluster barrier each CTA waits for exactly those incoming bulk copies.
// Only then is TMEM freed and, after a second cluster barrier, the CTA exits:
// no tensor-core operation, copy or remote write is in flight past that point.
//
// Building with -DMTV_TRACE records clock64() timestamps of the pipeline
// events of one CTA (chosen with mtv_trace_select, read with mtv_trace_read)
// and start/end times, SM and tile count of every CTA (mtv_trace_cta_read).
#include <math.h>

#include "mtv_internal.cuh"
#include "tc_ptx.cuh"

namespace mtv {

extern const int kTcRowTile = 128;
extern const int kTcKeyTile = 64;

namespace {

using namespace ptx;

constexpr int ROWS = 128;   // query rows per CTA pair
constexpr int NK = 64;      // keys per tile
#ifndef MTV_TC_STAGES
#define MTV_TC_STAGES 4  // shared memory holds four 36 KB stages next to the exchange buffers
#endif
constexpr int STAGES = MTV_TC_STAGES;  // gather pipeline depth
#ifndef MTV_TC_GATHER_WARPS
#define MTV_TC_GATHER_WARPS 2
#endif
constexpr int NPROD_WARPS = MTV_TC_GATHER_WARPS;
#ifndef MTV_TC_SOFTMAX_WARPS
#define MTV_TC_SOFTMAX_WARPS 4
#endif
constexpr int NSOFT_WARPS = MTV_TC_SOFTMAX_WARPS;  // 4 or 8: WPQ per TMEM lane quarter
constexpr int WPQ = NSOFT_WARPS / 4;       // softmax warps sharing one lane quarter (one row)
constexpr int NCOL = NK / WPQ;             // key columns per softmax warp
constexpr int OCOLS = 256 / WPQ;           // O columns per softmax warp (rescale, epilogue)
constexpr int XU = NCOL * 2 / 16;          // 16-byte units of one thread's quantised partial row
constexpr uint64_t kColMask = NCOL >= 64 ? ~0ull : ((1ull << NCOL) - 1ull);
constexpr int NTHREADS = 32 * (1 + NPROD_WARPS + NSOFT_WARPS);  // warp 0 MMA, then gather, then softmax
constexpr int KSTEPS2 = NK / 16;          // 4
constexpr float kRescaleLog2 = 8.0f;      // move the reference max only past 2^8 growth
constexpr float kQuantMagic = 12615680.0f;  // 1.5 * 2^23 + 2^15
constexpr long long kDrainCycles = 1ll << 31;  // bound of each wind-down wait (~1 s)
constexpr int kMaxKeysPerGatherWarp = (NK + NPROD_WARPS - 1) / NPROD_WARPS;
constexpr int kRopeGroups = (kMaxKeysPerGatherWarp + 7) / 8;  // rope copies: 8 keys x 4 lanes per instruction

constexpr uint32_t kChunkBytes = NK * 128;                       // 64 latent dims x 64 keys
constexpr uint32_t kRopeBytes = NK * 64;                          // 32 rope dims x 64 keys
constexpr uint32_t kStageBytes = 4 * kChunkBytes + kRopeBytes;    // 36 KB
constexpr uint32_t kOffStages = 0;
constexpr uint32_t kOffQRope = kOffStages + STAGES * kStageBytes;  // rope part of Q, 64B-swizzled
constexpr uint32_t kQRopeBytes = ROWS * 64;
// Partial-score exchange.  One region per softmax warp: its 32 rows x NCOL
// int16 (16-byte units swizzled), then one int8 step exponent per row, then
// one fp32 midpoint per row.  Two receive buffers (written by the peer) and
// two send buffers (staging for the bulk copies), each NSOFT_WARPS regions.
constexpr uint32_t kXRowBytes = NCOL * 2;
constexpr uint32_t kXOffExp = 32 * kXRowBytes;
constexpr uint32_t kXOffMid = kXOffExp + 32;
constexpr uint32_t kXRegion = kXOffMid + 32 * 4;
constexpr uint32_t kXBytes = NSOFT_WARPS * kXRegion;               // bytes completed per tile
constexpr uint32_t kOffRx = kOffQRope + kQRopeBytes;
constexpr uint32_t kOffTx = kOffRx + 2 * kXBytes;
constexpr uint32_t kOffVmask = kOffTx + 2 * kXBytes;                // [stage][8] key validity masks
constexpr uint32_t kVmaskBytes = STAGES * 8 * 8;
constexpr uint32_t kOffRowMax = kOffVmask + kVmaskBytes;          // [2 tiles][WPQ][128 rows] f32
constexpr uint32_t kRowMaxBytes = 2 * WPQ * ROWS * 4;
constexpr uint32_t kOffLsum = kOffRowMax + kRowMaxBytes;          // [WPQ][128 rows] f32
constexpr uint32_t kLsumBytes = 2 * WPQ * ROWS * 4;  // exact and bf16-rounded weight sums
constexpr uint32_t kOffBars = kOffLsum + kLsumBytes;
constexpr uint32_t kOffCtl = kOffBars + 256;
constexpr uint32_t kCtlBytes = 256;
constexpr uint32_t kSmemBytes = kOffCtl + kCtlBytes + 1024;  // + slack for 1 KB alignment

constexpr uint32_t kTmemO = 0, kTmemS = 256, kTmemQ = 320, kTmemP = 448;

enum : int {
  B_KV_FULL = 0, B_KV_EMPTY = STAGES, B_S_FULL = 2 * STAGES, B_S_FREE, B_P_FULL0, B_P_FULL1, B_O_READY0,
  B_O_READY1, B_Q_READY, B_SX_FULL0, B_SX_FULL1, B_FIN, B_QMAX, B_COUNT = B_QMAX + 4
};
static_assert(B_COUNT * 8 <= 256, "barrier area");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kOffQRope % 1024 == 0, "64B-swizzled operand alignment");
static_assert(NPROD_WARPS <= 8, "one 64-bit validity word per gather warp, 8 per stage");
static_assert((NSOFT_WARPS == 4 || NSOFT_WARPS == 8) && NCOL % 8 == 0 &&
                  (XU & (XU - 1)) == 0,
              "softmax column split");
static_assert(kXRegion % 16 == 0 && kOffRx % 16 == 0 && kOffTx % 16 == 0, "bulk copy alignment");

struct Ctl {
  uint32_t tmem_base;
  volatile int abort;           // set by a wait of this CTA or of the peer that gave up
  int armed;                    // score-exchange phases armed with the expected bytes
  int waited[NSOFT_WARPS];      // per softmax warp: exchange phases it saw complete
  int peer_sent[NSOFT_WARPS];   // written by the peer: score tiles each of its warps sent here
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

#ifdef MTV_TRACE
constexpr int kTraceTiles = 128, kTraceEvents = 16;
__device__ long long g_trace[4][kTraceTiles][kTraceEvents];
__device__ int g_trace_cta = 0;  // linear index (y * gridDim.x + x) of the CTA whose pipeline is traced
constexpr int kTraceCtas = 1 << 14;
__device__ long long g_cta_trace[kTraceCtas][4];  // per CTA: start ns, end ns, SM id, tiles
__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define MTV_TR(role, tile, ev)                                                                            \
  do {                                                                                                    \
    if (int(blockIdx.y * gridDim.x + blockIdx.x) == g_trace_cta && (tile) < kTraceTiles)              \
      g_trace[role][tile][ev] = clock64();                                                              \
  } while (0)
#else
#define MTV_TR(role, tile, ev) \
  do {                         \
  } while (0)
#endif

// Four normalised O values to global memory: fp32 partials or bf16 output.
__device__ __forceinline__ void store4(float* dst, float4 v) { *reinterpret_cast<float4*>(dst) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* dst, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// What a wait needs to give up: the flags of this CTA, the error word, the
// bound, and the cluster address of the peer's abort flag.
struct Waiter {
  Ctl* ctl;
  unsigned* err;
  long long limit;
  uint32_t peer_abort;
};

// Timeout: record it and stop both CTAs of the pair.
__device__ __noinline__ void give_up(Ctl* ctl, unsigned* err, uint32_t peer_abort) {
  ctl->abort = 1;
  st_cluster_u32(peer_abort, 1u);
  atomicOr(err, MTV_DEVERR_TIMEOUT);
}

// Bounded wait on a CTA barrier; false on timeout (after give_up) or abort.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctl* ctl, unsigned* err, long long limit,
                                      uint32_t peer_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ctl->abort) return false;
    if (clock64() - t0 > limit) {
      give_up(ctl, err, peer_abort);
      return false;
    }
  }
}

// Inline fast path: most waits find the phase already complete.
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, const Waiter& w) {
  return mbar_try_wait(bar, parity) || wait_bar(bar, parity, w.ctl, w.err, w.limit, w.peer_abort);
}

// Wind-down wait: ignores the abort flag; its own bound only guards against a
// broken device (it sets the timeout bit and returns false).
__device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity, unsigned* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kDrainCycles) {
      atomicOr(err, MTV_DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1) partial_tc_kernel(const Params P) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(gbase + kOffCtl);
  auto bar = [&](int i) { return base + kOffBars + 8u * uint32_t(i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int r = pair / P.grid_rows, rb = pair % P.grid_rows;
  const int split = blockIdx.y;
  if (threadIdx.x == 0) MTV_TR(1, kTraceTiles - 1, 0);
#ifdef MTV_TRACE
  const int cta_id = int(blockIdx.y * gridDim.x + blockIdx.x);
  if (threadIdx.x == 0 && cta_id < kTraceCtas) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_cta_trace[cta_id][0] = global_ns();
    g_cta_trace[cta_id][1] = 0;
    g_cta_trace[cta_id][2] = smid;
    g_cta_trace[cta_id][3] = -1;
  }
#endif
  const Req R = load_req(P, r);
  const int64_t rows_req = R.n * kHeads;
  if (int64_t(rb) * ROWS >= rows_req) return;  // both CTAs of the pair take this exit
  const int64_t k_begin = int64_t(split) * P.split_keys;
  if (split > 0 && k_begin >= R.keys) return;  // empty split: the combine never reads it
  const int64_t k_end = min(R.keys, k_begin + P.split_keys);
  const int T = int((k_end - k_begin + NK - 1) / NK);
#ifdef MTV_TRACE
  if (threadIdx.x == 0 && cta_id < kTraceCtas) g_cta_trace[cta_id][3] = T;
#endif
  uint64_t* vmask_all = reinterpret_cast<uint64_t*>(gbase + kOffVmask);  // [stage][8]

  // Slot of gather lane `lane` of warp `pw` for tile j (raw, checked at use).
  auto raw_slot_of = [&](int pw, int j) -> int64_t {
    int64_t v = -1;
    const int nmine = (NK - pw + NPROD_WARPS - 1) / NPROD_WARPS;
    if (lane < nmine && j < T) {
      const int64_t k = k_begin + int64_t(j) * NK + pw + NPROD_WARPS * lane;
      if (k < k_end) v = (k < R.p) ? P.kv_indices[R.kv_off + k] : P.out_cache_loc[R.q_off + (k - R.p)];
    }
    return v;
  };
  // The gather warps issue the index loads of their first two tiles before
  // the setup below, so that the load latency overlaps it.
  int64_t pre0 = -1, pre1 = -1;
  if (warp >= 1 && warp <= NPROD_WARPS) {
    pre0 = raw_slot_of(warp - 1, 0);
    pre1 = raw_slot_of(warp - 1, 1);
  }
  // Likewise the softmax warps load their rows of Q (this CTA's latent half
  // and rope part) with every load in flight at once; they store them after
  // the setup.  Rows past the request's end read as zeros.
  constexpr int kQChunks = 8 / WPQ;  // 16-column TMEM chunks per warp
  uint4 qpre[kQChunks][4], qrope[4];
  if (warp > NPROD_WARPS) {
    const int h0 = (warp - 1 - NPROD_WARPS) >> 2;
    const int64_t g0 = int64_t(rb) * ROWS + (warp & 3) * 32 + lane;
    const bool v0 = g0 < rows_req;
    const uint4* src = reinterpret_cast<const uint4*>(P.q + (R.q_off * kHeads + (v0 ? g0 : 0)) * kDQK);
#pragma unroll
    for (int i = 0; i < kQChunks; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        qpre[i][u] = v0 ? __ldg(src + (crank * 256 + 32 * (h0 + WPQ * i)) / 8 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      qrope[u] = (v0 && h0 == 0) ? __ldg(src + (512 + crank * 32) / 8 + u) : make_uint4(0u, 0u, 0u, 0u);
  }

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(B_KV_FULL + s), NPROD_WARPS * 33);  // 32 copy completions + 1 mask arrival per warp
      mbar_init(bar(B_KV_EMPTY + s), 1);
    }
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_S_FREE), NSOFT_WARPS);
    mbar_init(bar(B_P_FULL0), NSOFT_WARPS);
    mbar_init(bar(B_P_FULL1), NSOFT_WARPS);
    mbar_init(bar(B_O_READY0), 1);
    mbar_init(bar(B_O_READY1), 1);
    mbar_init(bar(B_Q_READY), NSOFT_WARPS);
    mbar_init(bar(B_SX_FULL0), 1);  // one local expect_tx arrival + the peer's bulk-copy bytes
    mbar_init(bar(B_SX_FULL1), 1);
    mbar_init(bar(B_FIN), 1);
    for (int qq = 0; qq < 4; ++qq) mbar_init(bar(B_QMAX + qq), WPQ);
    ctl->abort = 0;
    ctl->armed = 0;
    for (int w = 0; w < NSOFT_WARPS; ++w) ctl->waited[w] = ctl->peer_sent[w] = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&ctl->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // barriers and control blocks of both CTAs initialised before any remote access
  if (threadIdx.x == 0) MTV_TR(1, kTraceTiles - 1, 1);
  const uint32_t tmem = ctl->tmem_base;
  const Waiter W{ctl, P.err, P.wait_cycles, mapa(smem_u32(const_cast<int*>(&ctl->abort)), peer)};

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16_f32(128, NK, 0, 0);
      const uint32_t id2 = idesc_bf16_f32(128, 256, 0, 1);
      // Descriptors differ from a stage's base descriptor only in the start
      // address field (bits 0..13, address >> 4): shared-memory addresses stay
      // below 2^18, so adding an offset to the low word never carries out of
      // the field.  (Fewer instructions per MMA on the issuing thread.)
      auto desc_add = [](uint64_t d, uint32_t off) -> uint64_t {
        return (d & 0xFFFFFFFF00000000ull) | uint64_t(uint32_t(d) + (off >> 4));
      };
      const uint64_t rope_a0 = smem_desc(base + kOffQRope, 16, 512, kSwizzle64B);
      // GEMM1 of tile j: S = Q . K^T into the single S buffer.
      auto gemm1 = [&](int jj) {
        MTV_TR(0, jj, 1);
        fence_proxy_async_smem();  // cp.async wrote the stage through the generic proxy
        tc_fence_after();
        const uint32_t st = base + kOffStages + uint32_t(jj % STAGES) * kStageBytes;
        const uint64_t b0 = smem_desc(st, 16, 1024, kSwizzle128B);
        const uint64_t r0 = smem_desc(st + 4 * kChunkBytes, 16, 512, kSwizzle64B);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint64_t bd = desc_add(b0, uint32_t((kk >> 2) * kChunkBytes + (kk & 3) * 32));
          mma_ts(tmem + kTmemS, tmem + kTmemQ + kk * 8, bd, id1, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          mma_ss(tmem + kTmemS, desc_add(rope_a0, uint32_t(kk * 32)), desc_add(r0, uint32_t(kk * 32)), id1, 1u);
        }
        mma_commit(bar(B_S_FULL));
      };
      // GEMM2 of tile j: O += P . V, P from TMEM buffer j&1, V from the tile's stage.
      auto gemm2 = [&](int jj) {
        MTV_TR(0, jj, 2);
        tc_fence_after();
        const uint32_t st = base + kOffStages + uint32_t(jj % STAGES) * kStageBytes;
        const uint32_t pa = tmem + kTmemP + 32u * uint32_t(jj & 1);
        const uint64_t v0 = smem_desc(st, kChunkBytes, 1024, kSwizzle128B);
#pragma unroll
        for (int kk = 0; kk < KSTEPS2; ++kk) {
          const uint64_t bd = desc_add(v0, uint32_t(kk * 2048));
          mma_ts(tmem + kTmemO, pa + kk * 8, bd, id2, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(B_O_READY0 + (jj & 1)));
        mma_commit(bar(B_KV_EMPTY + jj % STAGES));
      };
      // Event-driven issue: GEMM1(j1) as soon as the softmax has read S(j1-1)
      // and its stage has landed; GEMM2(j2) as soon as P(j2) is in TMEM, and
      // first when both are ready (it frees a stage and a P buffer, and lets
      // the softmax rescale O sooner; measured 1-2 % faster than GEMM1 first).
      // The two streams never wait on each other's inputs, so a late stage does
      // not hold back the GEMM2 that frees an earlier one.  Tensor-core
      // operations of one thread run in issue order, and GEMM2(j) is only
      // issued after GEMM1(j).
      bool ok = wait_fast(bar(B_Q_READY), 0, W);
      int j1 = 0, j2 = 0;
      long long t_prog = clock64();
      while (ok && j2 < T) {
        bool did = false;
        if (j2 < j1 && mbar_test_wait(bar(B_P_FULL0 + (j2 & 1)), (j2 >> 1) & 1)) {
          gemm2(j2);
          ++j2;
          did = true;
        }
        if (j1 < T && (j1 == 0 || mbar_test_wait(bar(B_S_FREE), (j1 - 1) & 1)) &&
            mbar_test_wait(bar(B_KV_FULL + j1 % STAGES), (j1 / STAGES) & 1)) {
          MTV_TR(0, j1, 0);
          gemm1(j1);
          ++j1;
          did = true;
        }
        if (did) {
          t_prog = clock64();
        } else {
          if (ctl->abort) break;
          if (clock64() - t_prog > W.limit) {
            give_up(ctl, P.err, W.peer_abort);
            break;
          }
          __nanosleep(32);
        }
      }
      // Every MMA issued above has completed once B_FIN arrives (tensor-core
      // operations of one thread complete in order); waited for even after an
      // abort, since TMEM is freed below.
      mma_commit(bar(B_FIN));
      drain_wait(bar(B_FIN), 0, P.err);
    }
    __syncwarp();
  } else if (warp <= NPROD_WARPS) {
    // ------------------------------------------------------------ gather
    // Warp pw copies keys pw, pw + NPROD_WARPS, ... of each tile.  Lane i
    // holds the slot of the warp's i-th key, loaded two tiles ahead and only
    // checked when used, so index latency never stalls the warp.  Per key the
    // warp issues one 512-byte latent copy (32 lanes x 16 B), and per group
    // of 8 keys one copy of their 64-byte rope parts (4 lanes per key), into
    // the swizzled operand layout; an invalid slot is zero-filled (source
    // size 0).  Each lane then arrives on the stage's barrier when its own
    // copies land: the warp only waits for a free stage.
    const int pw = warp - 1;
    const int nmine = (NK - pw + NPROD_WARPS - 1) / NPROD_WARPS;
    // per-key swizzled destination offsets within a stage (same for every tile)
    uint32_t lat_off[kMaxKeysPerGatherWarp], rope_off[kRopeGroups];
#pragma unroll
    for (int i = 0; i < kMaxKeysPerGatherWarp; ++i) {
      const int kk = pw + NPROD_WARPS * i;
      lat_off[i] = uint32_t(lane >> 3) * kChunkBytes + kk * 128 + (((lane & 7) ^ (kk & 7)) << 4);
    }
#pragma unroll
    for (int g = 0; g < kRopeGroups; ++g) {
      const int kk = pw + NPROD_WARPS * (8 * g + (lane >> 2));
      rope_off[g] = 4 * kChunkBytes + kk * 64 + (((lane & 3) ^ ((kk >> 1) & 3)) << 4);
    }
    const unsigned char* pool_lat = reinterpret_cast<const unsigned char*>(P.kv_pool) + crank * 512 + lane * 16;
    const unsigned char* pool_rope =
        reinterpret_cast<const unsigned char*>(P.kv_pool) + 1024 + crank * 64 + (lane & 3) * 16;
    int64_t v0 = pre0, v1 = pre1;
    for (int j = 0; j < T; ++j) {
      const int s = j % STAGES;
      int slot = -1;  // checked slot of this lane's key (< 2^31 by the ABI contract)
      {
        const int64_t k = k_begin + int64_t(j) * NK + pw + NPROD_WARPS * lane;
        if (lane < nmine && k < k_end) {
          if (v0 >= 0 && v0 < P.num_slots) slot = int(v0);
          else atomicOr(P.err, MTV_DEVERR_SLOT_RANGE);
        }
      }
      v0 = v1;
      v1 = raw_slot_of(pw, j + 2);  // in flight until two iterations from now
      const int kk_l = pw + NPROD_WARPS * lane;
      const uint32_t vlo = __reduce_or_sync(0xffffffffu, (slot >= 0 && kk_l < 32) ? 1u << kk_l : 0u);
      const uint32_t vhi = __reduce_or_sync(0xffffffffu, (slot >= 0 && kk_l >= 32) ? 1u << (kk_l - 32) : 0u);
      if (j >= STAGES) {
        bool ok = wait_fast(bar(B_KV_EMPTY + s), ((j / STAGES) - 1) & 1, W);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (pw == 0 && lane == 0) MTV_TR(1, j, 0);
      const uint32_t st = base + kOffStages + uint32_t(s) * kStageBytes;
      const uint32_t fb = bar(B_KV_FULL + s);
      if (lane == 0) {
        vmask_all[s * 8 + pw] = (uint64_t(vhi) << 32) | vlo;
        mbar_arrive(fb);  // release: publishes this warp's mask
      }
#pragma unroll
      for (int i = 0; i < kMaxKeysPerGatherWarp; ++i) {
        if (i < nmine) {
          const int sl = __shfl_sync(0xffffffffu, slot, i);
          const int64_t row = int64_t(sl < 0 ? 0 : sl) * (kDQK * 2);
          cp_async_16_zfill(st + lat_off[i], pool_lat + row, sl >= 0 ? 16u : 0u);
        }
      }
#pragma unroll
      for (int g = 0; g < kRopeGroups; ++g) {
        const int i = 8 * g + (lane >> 2);  // this lane's key in the group (< 32)
        const int sl = __shfl_sync(0xffffffffu, slot, i);
        if (i < nmine) {
          const int64_t row = int64_t(sl < 0 ? 0 : sl) * (kDQK * 2);
          cp_async_16_zfill(st + rope_off[g], pool_rope + row, sl >= 0 ? 16u : 0u);
        }
      }
      cp_async_arrive_noinc(fb);
      if (pw == 0 && lane == 0) MTV_TR(1, j, 1);
    }
    cp_async_wait<0>();  // no copy may be in flight when the CTA exits
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int sw = warp - 1 - NPROD_WARPS;         // 0 .. NSOFT_WARPS-1
    const int q = warp & 3;                        // TMEM lane quarter this warp may access
    const int h = sw >> 2;                         // key columns [NCOL*h, +NCOL), O columns [OCOLS*h, +OCOLS)
    const int rr = q * 32 + lane;                  // row within the pair tile = TMEM lane
    const int64_t grow = int64_t(rb) * ROWS + rr;  // row within the request
    const bool valid = grow < rows_req;
    // Rows are valid in runs of 64 (one tree token), so a warp's 32 rows are
    // all valid or all past the request's end (the second half of a row block
    // of a request with an odd tree size).  Such a warp runs a short loop that
    // keeps the pipeline's protocol -- it sends its (unused) score region,
    // waits for the peer's, frees S and writes P = 0 -- and skips the softmax.
    const bool wvalid = __any_sync(0xffffffffu, valid);
    const int64_t ti = grow / kHeads;              // tree token of this row
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const int64_t out_row = R.q_off * kHeads + grow;  // (token, head) row of q/out/lse
    const uint32_t qbar = bar(B_QMAX + q);            // meeting point of the WPQ warps of this quarter
    float* rowmax = reinterpret_cast<float*>(gbase + kOffRowMax);  // [tile&1][h][row]
    float* lsum_s = reinterpret_cast<float*>(gbase + kOffLsum);    // [2][h][row]
    const bool tracer = (sw == 0 && lane == 0);
    const bool tracer2 = (sw == NSOFT_WARPS - 1 && lane == 0);
    // Scores stay in raw (unscaled) units; the scale enters once per element in
    // the exponent: p = 2^(x*c - m*c) with c = scale*log2(e).
    const float c = P.scale_log2;
    const float thr_raw = kRescaleLog2 / c;

    // Q half (loaded into registers before the setup): latent dims -> TMEM
    // (A operand, column j packs dims 2j, 2j+1; the warps of a quarter take
    // 16-column chunks in turn); rope dims -> shared memory in the 64B-swizzled
    // K-major layout (warp h = 0 writes them).
    {
#pragma unroll
      for (int i = 0; i < kQChunks; ++i) {
        uint32_t v[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          v[4 * u] = qpre[i][u].x; v[4 * u + 1] = qpre[i][u].y; v[4 * u + 2] = qpre[i][u].z; v[4 * u + 3] = qpre[i][u].w;
        }
        tmem_st16_sync(tmem + lane_off + kTmemQ + 16 * (h + WPQ * i), v);
      }
      if (h == 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 xq = qrope[u];
          st_shared_v4(base + kOffQRope + uint32_t(rr) * 64u + ((uint32_t(u) ^ ((uint32_t(rr) >> 1) & 3u)) << 4),
                       xq.x, xq.y, xq.z, xq.w);
        }
        fence_proxy_async_smem();  // read by the tensor core through the async proxy
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_Q_READY));
    }

    // Partial-score exchange, double-buffered: each warp stages the quantised
    // partial of tile j for its 32 rows in send buffer j&1 and bulk-copies the
    // region to the peer's receive buffer j&1, completing bytes on the peer's
    // barrier SX_FULL(j&1).  A warp sends tile j+1 only after SX_FULL(j)
    // completed and it has read tile j's values into registers.  SX_FULL(j)
    // completing means every peer warp has sent tile j, which each did only
    // after (a) reading tile j-1 -- the tile whose receive buffer (j+1)&1 tile
    // j+1 overwrites -- and (b) seeing SX_FULL(j-1) complete, i.e. our bulk
    // copies of tile j-1 had landed, so send buffer (j+1)&1 is free again.
    const int wreg = h * 4 + q;                               // region of this warp (same in both CTAs)
    const uint32_t x_lane = uint32_t(wreg) * kXRegion + uint32_t(lane) * kXRowBytes;
    const uint32_t x_exp = uint32_t(wreg) * kXRegion + kXOffExp + uint32_t(lane);
    const uint32_t x_mid = uint32_t(wreg) * kXRegion + kXOffMid + 4u * uint32_t(lane);
    // 16-byte unit swizzle: the rows sharing a 128-byte line get distinct unit orders
    const uint32_t x_sw = (uint32_t(lane) / uint32_t(128 / kXRowBytes)) & uint32_t(XU - 1);
    const uint32_t rx_peer = mapa(base + kOffRx, peer) + uint32_t(wreg) * kXRegion;
    const uint32_t peer_sx_full = mapa(bar(B_SX_FULL0), peer);  // + 8 for buffer 1
    // l: sum of the fp32 weights (gives the LSE); lr: sum of the same weights
    // rounded to bf16 as GEMM2 multiplies them (normalises O, so that the
    // rounding of a dominant weight cancels instead of scaling the output)
    float m_ref = -INFINITY, l = 0.f, lr = 0.f;
    bool alive = true;
    uint32_t s[NCOL];  // this CTA's partial scores of the tile being finished
    // wind-down bookkeeping: tiles this warp sent to the peer, exchange phases
    // it saw complete, and (tracer) phases armed with their expected bytes
    int nsent = 0, nwaited = 0, narmed = 0;

    // Load tile jn's partial scores from TMEM and send them to the peer as
    // NCOL 16-bit integers relative to their midpoint mid = (max + min)/2 with
    // a step 2^(k-15), where the half-range (max - min)/2 < 2^k (with a small
    // margin): u = rint((v - mid) * 2^(15-k)) + 2^15, 31 <= u <= 2^16 - 31.
    // The rounding is done by the adder: for |y| < 2^15, y + (1.5*2^23 + 2^15)
    // lands in [2^23, 2^24), where the float spacing is 1, and its low 16
    // mantissa bits are rint(y) + 2^15.  The receiver rebuilds 1.5*2^23 + u as float bits and
    // subtracts exactly; mid travels as an fp32 per row and is added per row
    // (in the row max and the exponent bias), never per value.
    auto fetch_and_send = [&](int jn) -> bool {
      bool ok = wait_fast(bar(B_S_FULL), jn & 1, W);
      if (!__all_sync(0xffffffffu, ok)) return false;
      if (tracer) MTV_TR(2, jn, 0);
      tc_fence_after();
      tmem_ld_sync(tmem + lane_off + kTmemS + NCOL * h, s);
      if (tracer) MTV_TR(2, jn, 6);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S_FREE));
      // (reductions run as independent chains: the min/max instructions are opaque to the compiler)
      float hi[2] = {-INFINITY, -INFINITY}, lo[2] = {INFINITY, INFINITY};
#pragma unroll
      for (int u = 0; u < NCOL; u += 2) {
        hi[(u >> 1) & 1] = max3(hi[(u >> 1) & 1], __uint_as_float(s[u]), __uint_as_float(s[u + 1]));
        lo[(u >> 1) & 1] = min3(lo[(u >> 1) & 1], __uint_as_float(s[u]), __uint_as_float(s[u + 1]));
      }
      const float vmax = fmaxf(hi[0], hi[1]), vmin = fminf(lo[0], lo[1]);
      const float mid = 0.5f * (vmax + vmin);
      // bound on |v - mid| over the block, with a 2^-10 margin for the roundings
      // of mid and of the subtractions: |y| = |v - mid| * 2^(15-k) < 2^15 - 31
      const float span = fmaxf(vmax - mid, mid - vmin) * (1.0f + 0x1p-10f);
      // span in [2^(k-1), 2^k) for normal span; 0 and subnormals give k <= -126
      int k = int((__float_as_uint(span) >> 23) & 0xffu) - 126;
      k = max(-100, min(k, 100));
      const float qs = __int_as_float((127 + 15 - k) << 23);  // 2^(15-k), exact
      const uint64_t qs2 = f2_pack(qs, qs), mg2 = f2_pack(kQuantMagic, kQuantMagic), nmid2 = f2_pack(-mid, -mid);
      const uint32_t tx = base + kOffTx + uint32_t(jn & 1) * kXBytes;
#pragma unroll
      for (int u = 0; u < XU; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c0 = 8 * u + 2 * e;
          float a, b;
          // v - mid is exact to 2^-24 of the half-range; the fma then rounds to the step
          const uint64_t d2 = f2_add(f2_pack(__uint_as_float(s[c0]), __uint_as_float(s[c0 + 1])), nmid2);
          f2_unpack(f2_fma(d2, qs2, mg2), a, b);
          w[e] = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x5410);
        }
        st_shared_v4(tx + x_lane + ((uint32_t(u) ^ x_sw) << 4), w[0], w[1], w[2], w[3]);
      }
      st_shared_f32(tx + x_mid, mid);
      st_shared_u8(tx + x_exp, uint32_t(k));
      fence_proxy_async_smem();  // the bulk copy reads the staging through the async proxy
      __syncwarp();
      if (lane == 0)
        bulk_copy_to_peer(rx_peer + uint32_t(jn & 1) * kXBytes, tx + uint32_t(wreg) * kXRegion, kXRegion,
                          peer_sx_full + 8u * uint32_t(jn & 1));
      ++nsent;
      if (tracer) MTV_TR(2, jn, 1);
      if (tracer2) MTV_TR(3, jn, 1);
      return true;
    };

    if (!wvalid) {
      // Rows past the request's end (see wvalid): the same barrier and copy
      // sequence as the loop below, without the arithmetic.
      auto idle_send = [&](int jn) -> bool {
        bool ok = wait_fast(bar(B_S_FULL), jn & 1, W);
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc_fence_after();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B_S_FREE));
          bulk_copy_to_peer(rx_peer + uint32_t(jn & 1) * kXBytes,
                            base + kOffTx + uint32_t(jn & 1) * kXBytes + uint32_t(wreg) * kXRegion, kXRegion,
                            peer_sx_full + 8u * uint32_t(jn & 1));
        }
        ++nsent;
        return true;
      };
      if (tracer) mbar_arrive_expect_tx(bar(B_SX_FULL0), kXBytes);  // tile 0
      narmed = 1;
      alive = idle_send(0);
      const uint32_t zero[NCOL / 2] = {};
      for (int j = 0; alive && j < T; ++j) {
        if (j + 1 < T) {
          if (tracer) mbar_arrive_expect_tx(bar(B_SX_FULL0 + ((j + 1) & 1)), kXBytes);
          narmed = j + 2;
        }
        bool ok = wait_fast(bar(B_SX_FULL0 + (j & 1)), (j >> 1) & 1, W);
        if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
        nwaited = j + 1;
        if (j + 1 < T && !idle_send(j + 1)) { alive = false; break; }
        if (j >= 2) {  // P buffer j&1 was last read by GEMM2(j-2)
          ok = wait_fast(bar(B_O_READY0 + (j & 1)), ((j - 2) >> 1) & 1, W);
          if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
        }
        tc_fence_after();
        tmem_st_sync(tmem + lane_off + kTmemP + 32 * (j & 1) + (NCOL / 2) * h, zero);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_P_FULL0 + (j & 1)));
      }
    } else {
    if (tracer) mbar_arrive_expect_tx(bar(B_SX_FULL0), kXBytes);  // tile 0
    narmed = 1;
    alive = fetch_and_send(0);
    for (int j = 0; alive && j < T; ++j) {
      // tile j+1's bytes land in buffer (j+1)&1, whose previous phase (tile j-1) is complete
      if (j + 1 < T) {
        if (tracer) mbar_arrive_expect_tx(bar(B_SX_FULL0 + ((j + 1) & 1)), kXBytes);
        narmed = j + 2;
      }
      bool ok = wait_fast(bar(B_SX_FULL0 + (j & 1)), (j >> 1) & 1, W);
      if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
      nwaited = j + 1;
      if (tracer) MTV_TR(2, j, 2);
      if (tracer2) MTV_TR(3, j, 2);
      // full scores of this warp's columns, less the peer's block midpoint xmid:
      // own exact partial + peer's partial relative to xmid
      float x[NCOL], xmid;
      {
        const unsigned char* rxb = gbase + kOffRx + (j & 1) * kXBytes;
        const int kp = *reinterpret_cast<const signed char*>(rxb + x_exp);
        xmid = *reinterpret_cast<const float*>(rxb + x_mid);
        const float dq = __int_as_float((127 - 15 + kp) << 23);  // 2^(k-15)
        const uint64_t dq2 = f2_pack(dq, dq), nmg2 = f2_pack(-kQuantMagic, -kQuantMagic);
        const uint4* row = reinterpret_cast<const uint4*>(rxb + x_lane);
#pragma unroll
        for (int u = 0; u < XU; ++u) {
          const uint4 v = row[u ^ x_sw];
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c0 = 8 * u + 2 * e;
            const float flo = __uint_as_float(__byte_perm(wv[e], 0x4B40u, 0x5410));  // 1.5*2^23 + u_lo
            const float fhi = __uint_as_float(__byte_perm(wv[e], 0x4B40u, 0x5432));  // 1.5*2^23 + u_hi
            const uint64_t t2 = f2_add(f2_pack(flo, fhi), nmg2);                     // exact integers
            f2_unpack(f2_fma(t2, dq2, f2_pack(__uint_as_float(s[c0]), __uint_as_float(s[c0 + 1]))), x[c0],
                      x[c0 + 1]);
          }
        }
      }
      // x now holds every value read from buffer j&1 (the empty asm orders the
      // reads before the send below), so tile j+1 may be sent into buffer (j+1)&1.
#pragma unroll
      for (int cc = 0; cc < NCOL; ++cc) asm volatile("" : "+f"(x[cc]));
      if (tracer) MTV_TR(2, j, 7);
      if (j + 1 < T && !fetch_and_send(j + 1)) { alive = false; break; }

      // tree mask (raw units; masked -> -inf)
      const int sidx = j % STAGES;
      ok = wait_fast(bar(B_KV_FULL + sidx), (j / STAGES) & 1, W);
      if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
      if (tracer) MTV_TR(2, j, 8);
      uint64_t vm = 0;  // OR of the gather warps' masks (exactly NPROD_WARPS words are written)
      {
        const ulonglong2* vp = reinterpret_cast<const ulonglong2*>(vmask_all + sidx * 8);
#pragma unroll
        for (int w2 = 0; w2 < NPROD_WARPS / 2; ++w2) {
          const ulonglong2 a = vp[w2];
          vm |= a.x | a.y;
        }
        if (NPROD_WARPS & 1) vm |= vmask_all[sidx * 8 + NPROD_WARPS - 1];
      }
      const uint64_t vbits = (vm >> (NCOL * h)) & kColMask;
      const int64_t kt = k_begin + int64_t(j) * NK + NCOL * h;  // key of this warp's first column
      if (!(valid && vbits == kColMask && kt + NCOL <= R.p)) {  // not an all-prefix, all-valid tile
#pragma unroll
        for (int cc = 0; cc < NCOL; ++cc) {
          const int64_t k = kt + cc;
          bool vis = valid && ((vbits >> cc) & 1ull);
          if (vis && k >= R.p) vis = tree_visible(P, R, ti, k - R.p);
          if (!vis) x[cc] = -INFINITY;
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int cc = 0; cc < NCOL; cc += 2) mx[(cc >> 1) & 3] = max3(mx[(cc >> 1) & 3], x[cc], x[cc + 1]);
      float mt = max3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) + xmid;  // -inf stays -inf
      if constexpr (WPQ > 1) {
        rowmax[((j & 1) * WPQ + h) * ROWS + rr] = mt;
        if (tracer) MTV_TR(2, j, 9);
        if (tracer2) MTV_TR(3, j, 9);
        // combine the tile max of the WPQ warps of this row (bounded mbarrier meeting)
        __syncwarp();
        if (lane == 0) mbar_arrive(qbar);
        ok = wait_fast(qbar, j & 1, W);
        if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
#pragma unroll
        for (int hh = 0; hh < WPQ; ++hh) mt = fmaxf(mt, rowmax[((j & 1) * WPQ + hh) * ROWS + rr]);
      }
      if (tracer) MTV_TR(2, j, 3);
      if (tracer2) MTV_TR(3, j, 3);

      const float m_new = fmaxf(m_ref, mt);
      const bool move = (m_new > m_ref + thr_raw) || (m_ref == -INFINITY && m_new != -INFINITY);
      const float fac = move ? ex2((m_ref - m_new) * c) : 1.f;  // ex2(-inf) = 0
      if (move) {
        l *= fac;
        lr *= fac;
        m_ref = m_new;
      }
      // exponent c*(x + xmid - m_ref): the midpoint enters through the bias
      const float nb = (m_ref == -INFINITY) ? 0.f : (xmid - m_ref) * c;
      const uint64_t c2 = f2_pack(c, c), nb2 = f2_pack(nb, nb);
      uint64_t ls[2], lsr[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) ls[i] = lsr[i] = f2_pack(0.f, 0.f);
      uint32_t pk[NCOL / 2];
#pragma unroll
      for (int u = 0; u < NCOL / 2; ++u) {
        float e0, e1;
        f2_unpack(f2_fma(f2_pack(x[2 * u], x[2 * u + 1]), c2, nb2), e0, e1);
        const float p0 = ex2(e0), p1 = ex2(e1);
        ls[u & 1] = f2_add(ls[u & 1], f2_pack(p0, p1));
        const __nv_bfloat162 b = __floats2bfloat162_rn(p0, p1);  // p0 in the low half
        pk[u] = *reinterpret_cast<const uint32_t*>(&b);
        lsr[u & 1] = f2_add(lsr[u & 1], f2_pack(__uint_as_float(pk[u] << 16), __uint_as_float(pk[u] & 0xffff0000u)));
      }
      {
        float a0, a1, b0, b1;
        f2_unpack(f2_add(ls[0], ls[1]), a0, a1);
        f2_unpack(f2_add(lsr[0], lsr[1]), b0, b1);
        l += a0 + a1;
        lr += b0 + b1;
      }

      if (tracer) MTV_TR(2, j, 10);
      // P buffer j&1 was last read by GEMM2(j-2); O may only be rescaled once
      // GEMM2(j-1) has finished accumulating into it.
      if (j >= 2) {
        ok = wait_fast(bar(B_O_READY0 + (j & 1)), ((j - 2) >> 1) & 1, W);
        if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
      }
      if (j >= 1 && __any_sync(0xffffffffu, move)) {  // warp-uniform TMEM read-modify-write of this warp's O columns
        ok = wait_fast(bar(B_O_READY0 + ((j - 1) & 1)), ((j - 1) >> 1) & 1, W);
        if (!__all_sync(0xffffffffu, ok)) { alive = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = OCOLS * h; c0 < OCOLS * h + OCOLS; c0 += 32) {
          uint32_t v[32];
          tmem_ld32_sync(tmem + lane_off + kTmemO + c0, v);
#pragma unroll
          for (int u = 0; u < 32; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) * fac);
          tmem_st32_sync(tmem + lane_off + kTmemO + c0, v);
        }
      }
      tc_fence_after();
      if (tracer) MTV_TR(2, j, 4);
      tmem_st_sync(tmem + lane_off + kTmemP + 32 * (j & 1) + (NCOL / 2) * h, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL0 + (j & 1)));
      if (tracer) MTV_TR(2, j, 5);
      if (tracer2) MTV_TR(3, j, 5);
    }

    if (tracer) MTV_TR(2, kTraceTiles - 1, 0);
    // epilogue: normalised O columns of this warp (+ LSE from CTA 0, warp h = 0)
    if (alive) {
      bool ok = wait_fast(bar(B_O_READY0 + ((T - 1) & 1)), ((T - 1) >> 1) & 1, W);
      alive = __all_sync(0xffffffffu, ok);
    }
    // the row's WPQ partial sums meet in shared memory
    if (alive) {
      lsum_s[h * ROWS + rr] = l;
      lsum_s[(WPQ + h) * ROWS + rr] = lr;
      __syncwarp();
      if (lane == 0) mbar_arrive(qbar);
      // the loop used one phase of this barrier per tile when WPQ > 1
      bool ok = wait_fast(qbar, WPQ > 1 ? (T & 1) : 0, W);
      alive = __all_sync(0xffffffffu, ok);
    }
    if (alive) {
      float tot = 0.f, totr = 0.f;
#pragma unroll
      for (int hh = 0; hh < WPQ; ++hh) {
        tot += lsum_s[hh * ROWS + rr];
        totr += lsum_s[(WPQ + hh) * ROWS + rr];
      }
      tc_fence_after();
      const float inv = totr > 0.f ? 1.f / totr : 0.f;
      // Normalised O columns go through shared memory so that the global
      // stores are row-contiguous: each thread holds one row, but a warp
      // stores two rows x 256 bytes per instruction.  The staging uses the
      // KV stage area, free once GEMM2(T-1) (the last tensor-core operation)
      // has completed; 16-byte units are XOR-swizzled by row (conflict-free).
      const uint32_t stg = base + kOffStages + uint32_t(sw) * (32u * OCOLS * 4u);  // 32 rows x OCOLS f32
      constexpr int kLdCols = OCOLS >= 64 ? 64 : 32;  // columns per TMEM load
#pragma unroll 1
      for (int c0 = 0; c0 < OCOLS; c0 += kLdCols) {
        uint32_t v[kLdCols];
        tmem_ld_sync(tmem + lane_off + kTmemO + OCOLS * h + c0, v);
#pragma unroll
        for (int u = 0; u < kLdCols / 4; ++u) {
          const uint32_t unit = uint32_t(c0 / 4 + u);
          st_shared_v4(stg + uint32_t(lane) * (OCOLS * 4u) + ((unit ^ (uint32_t(lane) & 15u)) << 4),
                       __float_as_uint(__uint_as_float(v[4 * u]) * inv),
                       __float_as_uint(__uint_as_float(v[4 * u + 1]) * inv),
                       __float_as_uint(__uint_as_float(v[4 * u + 2]) * inv),
                       __float_as_uint(__uint_as_float(v[4 * u + 3]) * inv));
        }
      }
      __syncwarp();
      constexpr int kUnits = OCOLS / 4;  // 16-byte units per staged row
      static_assert(kUnits % 32 == 0, "whole 512-byte row segments per warp");
      {
        // The warp's 32 rows are all valid here (see wvalid): row rl of the
        // warp is output row out_row - lane + rl.  Lane i stores units i,
        // i + 32, ... of each row: 512 contiguous bytes (fp32) or 256 (bf16)
        // per warp instruction.  Rows are unrolled by 8 so that the shared
        // loads of several rows are in flight before their stores.
        const int64_t row0 = out_row - lane;
        const int col = int(crank) * 256 + OCOLS * h + 4 * lane;
        auto store_rows = [&](auto* dst) {
#pragma unroll 8
          for (int rl = 0; rl < 32; ++rl) {
            const uint32_t src = stg + uint32_t(rl) * (OCOLS * 4u) + ((uint32_t(lane) ^ uint32_t(rl & 15)) << 4);
#pragma unroll
            for (int hf = 0; hf < kUnits / 32; ++hf) {
              const float4 val = ld_shared_f4(src + hf * 512);
              store4(dst + rl * kDLat + hf * 128, val);
            }
          }
        };
        if (P.nsplit == 1) store_rows(P.out + row0 * kDLat + col);
        else store_rows(P.part_o + (int64_t(split) * P.total_q_max * kHeads + row0) * kDLat + col);
      }
      if (valid && crank == 0 && h == 0) {
        const float lse = tot > 0.f ? (m_ref * c + __log2f(tot)) * kLn2 : -INFINITY;
        if (P.nsplit == 1) P.lse[out_row] = lse;
        else P.part_lse[int64_t(split) * P.total_q_max * kHeads + out_row] = lse;
      }
    }
    }
    // Wind-down bookkeeping (also after an abort): the peer learns how many
    // score tiles this warp sent it; the tracer records the armed phases.
    if (lane == 0) {
      ctl->waited[wreg] = nwaited;
      st_cluster_u32(mapa(smem_u32(&ctl->peer_sent[wreg]), peer), uint32_t(nsent));
    }
    if (tracer) ctl->armed = narmed;
  }

  // ---------------------------------------------------------------- wind-down
  // Every role has left its loop: the MMA issuer saw its last MMA complete,
  // the gather warps their copies.  The first cluster barrier publishes the
  // peer's sent counts and guarantees that every bulk copy into this CTA has
  // been issued.  Thread 0 then waits for exactly those bytes: phases from the
  // first one no warp saw complete, each armed (or its arming corrected) with
  // the bytes of the peer warps that sent that tile.  A warp sends tile j+1
  // only after seeing tile j arrive, so at most two tiles are outstanding and
  // they use different buffers.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();
  if (threadIdx.x == 0) {
    int j = 0;
    for (int w = 0; w < NSOFT_WARPS; ++w) j = max(j, ctl->waited[w]);
    for (;; ++j) {
      int senders = 0;
      for (int w = 0; w < NSOFT_WARPS; ++w) senders += ctl->peer_sent[w] > j ? 1 : 0;
      if (senders == 0) break;
      const uint32_t b = bar(B_SX_FULL0 + (j & 1));
      const uint32_t bytes = uint32_t(senders) * kXRegion;
      if (j < ctl->armed) {
        if (bytes < kXBytes) mbar_complete_tx(b, kXBytes - bytes);  // copies that will never come
      } else {
        mbar_arrive_expect_tx(b, bytes);
      }
      if (!drain_wait(b, (j >> 1) & 1, P.err)) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) MTV_TR(2, kTraceTiles - 1, 2);
  if (warp == 0) tmem_dealloc(tmem, 512);
  cluster_sync();  // both CTAs have received everything sent to them
  if (threadIdx.x == 0) MTV_TR(2, kTraceTiles - 1, 3);
#ifdef MTV_TRACE
  if (threadIdx.x == 0 && cta_id < kTraceCtas) g_cta_trace[cta_id][1] = global_ns();
#endif
}

}  // namespace

// Split count for the tensor-core kernel: fill the SM pairs in whole waves
// while keeping the fp32 partial traffic of the combine small.
int choose_nsplit_tc(int num_sms, int64_t pairs_per_split, int64_t max_keys, int64_t rows_total) {
  if (pairs_per_split <= 0) return 1;
  const double slots = double(num_sms / 2);
  const double t_key_us = 0.02;     // one 64-key tile costs ~1.3 us per pair; per key
  const double t_fixed_us = 4.0;    // launch, Q load, pipeline fill, epilogue
  const double hbm_bytes_per_us = 6.0e6;
  int best = 1;
  double best_t = 1e30;
  for (int ns = 1; ns <= 64; ++ns) {
    const double keys = double(((max_keys + ns - 1) / ns + NK - 1) / NK * NK);
    if (ns > 1 && keys * (ns - 1) >= double(max_keys) + NK) break;  // last split would be empty
    const double waves = ceil(double(pairs_per_split) * ns / slots);
    double t = waves * (keys * t_key_us + t_fixed_us);
    if (ns > 1) t += double(ns) * double(rows_total) * kDLat * 4.0 * 2.0 / hbm_bytes_per_us + 2.0;
    if (t < best_t * 0.98) {
      best_t = t;
      best = ns;
    }
  }
  return best;
}

cudaError_t prepare_partial_tc() {
  return cudaFuncSetAttribute(partial_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
}

cudaError_t launch_partial_tc(const Params& P, cudaStream_t st) {
  const int64_t pairs = int64_t(P.bs) * P.grid_rows;
  if (pairs == 0) return cudaSuccess;
  dim3 grid(unsigned(2 * pairs), unsigned(P.nsplit));
  partial_tc_kernel<<<grid, NTHREADS, kSmemBytes, st>>>(P);
  return cudaGetLastError();
}

}  // namespace mtv

#ifdef MTV_TRACE
extern "C" int mtv_trace_read(void* host, size_t bytes) {
  if (bytes > sizeof(mtv::g_trace)) bytes = sizeof(mtv::g_trace);
  return cudaMemcpyFromSymbol(host, mtv::g_trace, bytes) == cudaSuccess ? 0 : -7;
}
extern "C" int mtv_trace_select(int cta) {
  return cudaMemcpyToSymbol(mtv::g_trace_cta, &cta, sizeof cta) == cudaSuccess ? 0 : -7;
}
extern "C" int mtv_trace_cta_read(void* host, size_t bytes) {
  if (bytes > sizeof(mtv::g_cta_trace)) bytes = sizeof(mtv::g_cta_trace);
  return cudaMemcpyFromSymbol(host, mtv::g_cta_trace, bytes) == cudaSuccess ? 0 : -7;
}
extern "C" int mtv_trace_clear() {
  static long long zeros[4 * mtv::kTraceTiles * mtv::kTraceEvents];
  return cudaMemcpyToSymbol(mtv::g_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : -7;
}
#endif
