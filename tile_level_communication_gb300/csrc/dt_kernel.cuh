// Persistent, warp-specialised tcgen05 GEMM with the chunk-centric AllGather,
// ReduceScatter / AllReduce or AllToAll fused in.
//
// One CTA per SM, 8 warps; CL CTAs per cluster share a tile of CL x 128 rows (CL = 1: one
// CTA, tcgen05 cta_group::1; CL = 2: a CTA pair, cta_group::2):
//   warp 0      TMA producer: per tile, waits (bounded) for the ready flags of the chunks
//               this CTA's rows live in, then streams A / B k-blocks into a 4- or 6-stage
//               ring (a pair's stages complete on its even CTA's barriers).
//   warp 1      MMA issuer (one thread; the even CTA of a pair): tcgen05.mma 128x256x16 or
//               256x256x16 into one of two TMEM accumulators; allocates / frees TMEM.
//   warps 2-3   chunk transfer workers (AllGather, in-kernel backends): copy chunk pieces
//               from the rank shards into the gather buffer (TMA bulk or 16-byte ld/st)
//               and release each chunk's ready flag when its last piece has landed.
//   warps 4-7   epilogue: TMEM -> registers -> global.  AllGather: bf16 / fp32 C.
//               ReduceScatter / AllReduce: per (chunk piece, column tile) unit the
//               partial is folded into an fp32 running sum in the fixed source order, or
//               parked until its turn.  AllToAll: the tile's rows go straight into the
//               destination's block, then the chunk's count of stored tiles is notified.
//
// Sources: AutoOverlap page sections 4-5 (chunks, per-chunk waits inserted before the
// consuming tile, copy engine / TMA / ld-st lowerings with global-memory signals);
// Triton-distributed talk (notify / wait pairs, pull for AllGather, push for
// ReduceScatter); DITRON page section 3.2 (rank-aware tile order, see dt_plan.cuh).
#pragma once

#include <cuda_bf16.h>

#include "dt_plan.cuh"
#include "dt_ptx.cuh"

namespace dt {

constexpr int kBM = 128;                 // rows of A per CTA (a CTA pair's tile has 256)
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kThreads = 256;
constexpr int kAStage = kBM * kBK * 2;   // 16 KB: 128 rows x 64 bf16, 128-byte swizzle
constexpr int kBSlab = kBK * 64 * 2;     // 8 KB: 64 k-rows x 64 bf16 columns
// Operand ring per CTA: one CTA per tile stages all 256 columns of B (4 slabs, 32 KB) in 4
// stages; a CTA pair splits them (2 slabs, 16 KB each) and affords 6 stages next to the 32 KB
// staging buffers.
__host__ __device__ constexpr int stages(bool pair) { return pair ? 6 : 4; }
__host__ __device__ constexpr int b_slabs(bool pair) { return pair ? 2 : 4; }
__host__ __device__ constexpr int b_stage_bytes(bool pair) { return b_slabs(pair) * kBSlab; }
constexpr int kCopyBuf = 16384;          // TMA bulk copy staging, two buffers
constexpr int kTmemCols = 512;           // two 128x256 fp32 accumulators
constexpr int kMaxW = 16;
constexpr int kReadyBitsWords = 128;     // producer's cache of seen chunk flags (4096)
constexpr int kMiscBytes = 1024;

enum CopyMode : int { kCopyNone = 0, kCopyTma = 1, kCopyLdst = 2 };
// Which collective is fused: AllGather (gather mode, one A and B), ReduceScatter /
// AllReduce (scatter mode by rows, per-rank A_q and B_q), AllToAll (scatter mode by
// columns, per-rank A_q and B_q with each rank's rows tiled on their own).
enum OpKind : int { kOpAG = 0, kOpRS = 1, kOpA2A = 2 };

enum DevCode : uint32_t {
  kDevOk = 0,
  kDevTimeoutFlag = 1,   // a chunk's ready flag did not flip in time
  kDevTimeoutPipe = 2,   // a pipeline mbarrier did not complete in time
  kDevBadTile = 3,       // a tile id from the plan was out of range (tile skipped)
};

// Dynamic shared memory of a kernel instance: alignment slack, the operand ring, two 16 KiB
// staging buffers (AllGather: the co-located TMA transfer, else C's boxes on their way to a
// TMA store; ReduceScatter: running-sum tiles; AllToAll: out_h's boxes), flags.
// cl: CTAs per cluster (1: one CTA per 128-row tile; 2: a CTA pair per 256-row tile)
__host__ __device__ constexpr int kernel_smem_bytes(int cl) {
  return 1024 + stages(cl > 1) * (kAStage + b_stage_bytes(cl > 1)) + 2 * kCopyBuf + kMiscBytes;
}

struct KParams {
  CUtensorMap tmA[kMaxW];  // AG: [0] = gather buffer, [1] = own shard; RS / A2A: A_q
  CUtensorMap tmB[kMaxW];  // AG: [0] = B; RS / A2A: B_q
  CUtensorMap tmAcc;       // RS: running sums, fp32 [M][N], 32 x 128 boxes
  CUtensorMap tmPark;      // RS: park slots, fp32 [W (W-1) M/W][N], 32 x 128 boxes
  CUtensorMap tmOut[kMaxW];  // RS: out[s]; AR: out[r]; 32 x 128 boxes (bf16 dense rows, or
                             // fp32 in the running sums' 128-byte-swizzled layout)
  const uint8_t* shard[kMaxW];
  void* out[kMaxW];        // AG: out[0] = C; RS: out[s] ([M/W][N]); AR: out[r] ([M][N]);
                           // A2A: out[h] ([M][N/W]), or the ranks' own Y_q in the baseline
  uint8_t* gather;
  float* recv;             // RS: running sums [M][N] fp32, then the park slots
  uint32_t* ready;         // AG: per chunk, = epoch once landed; A2A: per (h, q, j), = epoch
                           // once every tile of that chunk has been stored
  uint32_t* pieces_done;   // AG: per chunk piece counter (back to 0 after the chunk)
  uint32_t* unit_cnt;      // RS: per (m-tile, chunk piece, column tile) arrival counter;
                           // A2A: per (h, q, j) count of stored tiles (back to 0 when done)
  const int32_t* order;    // tile order written by the prepare kernel
  uint32_t* err;           // 4 words: code, site, detail0, detail1
  unsigned long long* tag; // workspace layout tag; written at exit when no error was seen
  unsigned long long tag_value;
  Geom g;
  int64_t lda_src;         // AG: elements between shard rows
  int64_t ld_gather;       // AG: elements between gather rows
  int64_t ldc;
  int64_t row_lo, row_hi;  // rows handled: [0, M) fused; one window in the baselines
  int32_t Tm, KB, T;       // m-tiles in the window, k-blocks, tiles in the launch
  int32_t pieces_max;      // RS: most chunks one m-tile's rows touch (counter stride)
  int32_t ar_copies;       // 0: ReduceScatter; > 0: AllReduce into out[0 .. ar_copies-1]
  int32_t act;             // AG epilogue activation: 0 none, 1 GELU (tanh form), 2 SiLU
  int32_t own_in_place;    // AG: the own rank's tiles read its shard in place (tmA[1]) and
                           // its chunks are not transferred (its block is tile-aligned)
  int32_t copy_ctas;       // AG in-kernel transfer: CTAs 0..copy_ctas-1 only move chunks
                           // (dedicated SMs); 0: transfer warps inside every compute CTA
  int32_t plain;           // 1: identity order, no flags, no arrival counting
  int32_t a2a_step;        // A2A baseline launch: step d, every rank q computes destination
                           // (q + d + 1) mod W into out[q]; -1 in the fused kernel
  int32_t wait_flags;      // AG: the producer waits on ready flags
  uint32_t epoch;
  uint64_t timeout_ns;
  // in-kernel chunk transfer (AG)
  int64_t row_bytes;       // K * 2
  int32_t rows_per_piece;  // > 0: whole rows per piece; 0: a row is split in segments
  int32_t segs_per_row;
  int32_t pieces_full;     // pieces of a chunk with Cr rows
  int32_t pieces_last;     // pieces of the last chunk of a rank
  int32_t src_rows_contig; // shard rows are back to back (lda == K)
  int32_t drop_chunk;      // failure-detection testing: chunk the host told the in-kernel
                           // transfer to leave out (its flag never flips); -1: none
  int32_t l2_hints;        // ReduceScatter / AllReduce L2 cache policies: bit 0, running sums,
                           // park slots and final sums stream through L2 (evict first); bit 1,
                           // B_q's k-blocks stay (evict last)
  unsigned long long* trace;  // AG debug timeline (global timer, ns), or null; see trace_*
  int32_t c_tma;           // AG: C leaves through the staging buffers as TMA stores (tmOut[0],
                           // 32-column boxes clipped at M and N); A2A: out_h does (tmOut[h], 3-D
                           // [W][M/W][N/W], clipped at each source's rows); 0: per-thread rows
  int32_t a_from_shards;   // AG: each tile's A rows are loaded from the owning shard (tmA[s])
  int32_t ded_bufs;        // TMA buffers per worker on a dedicated transfer CTA: 1 to 4
  int32_t rot;             // per-wave rotation of the CTAs' slots in the tile order (pos_at)
  int32_t piece_bytes;     // bytes of one transfer piece and of one TMA worker buffer (a
                           // multiple of 16; kCopyBuf, or up to 2 * kCopyBuf on dedicated
                           // transfer CTAs)
  int32_t rs_reduce;       // ReduceScatter / AllReduce: a source between the first and the last
                           // folds its partial into the running sum with a TMA reduce-add (1)
                           // rather than a load, an add and a store (0)
};

// AG debug timeline, in 64-bit words: [0] first CTA start (min), [1] last CTA exit (max),
// [2] time the producers spent waiting for ready flags (sum over waits), [3] waits that had to
// wait; then per chunk c: [4 + 3c] release of its ready flag by the in-kernel transfer (min),
// [5 + 3c] first wait that found it missing began (min), [6 + 3c] first consumer passed its
// flag (min).  The host fills the min words with all ones and the others with zero.
constexpr int kTraceHead = 4;
__device__ __forceinline__ void trace_min(unsigned long long* tr, int64_t w) {
  if (tr != nullptr) atomicMin(tr + w, static_cast<unsigned long long>(globaltimer_ns()));
}

struct SmemLayout {
  uint8_t* a;
  uint8_t* b;
  uint8_t* copy;
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  volatile int* unit_flag;
  volatile int* vote;      // [2][4]
  volatile uint32_t* last_mask;  // RS: pieces of the current tile folded in order [4]
  volatile int8_t* chain;        // RS: per piece, first parked partial this tile folds (-1)
  uint32_t* ready_bits;
  int ns;  // pipeline stages
  // barrier slots: full[ns], empty[ns], tfull[2], tempty[2], copyb[2], fin (at most 21); on a
  // dedicated transfer CTA all 32 slots belong to its copy workers
  __device__ uint32_t full(int s) const { return smem_u32(bars + s); }
  __device__ uint32_t empty(int s) const { return smem_u32(bars + ns + s); }
  __device__ uint32_t tfull(int a) const { return smem_u32(bars + 2 * ns + a); }
  __device__ uint32_t tempty(int a) const { return smem_u32(bars + 2 * ns + 2 + a); }
  __device__ uint32_t copyb(int b) const { return smem_u32(bars + 2 * ns + 4 + b); }
  __device__ uint32_t fin() const { return smem_u32(bars + 2 * ns + 6); }
};

__device__ __forceinline__ void raise_error(const KParams& p, uint32_t code, uint32_t site,
                                            uint32_t d0, uint32_t d1) {
  if (atomicCAS(p.err, 0u, code) == 0u) {
    p.err[1] = site;
    p.err[2] = d0;
    p.err[3] = d1;
    __threadfence();
  }
}

// Bounded wait on an mbarrier phase.  On timeout records the error, raises the CTA's abort
// flag and returns false; returns false at once when another role has aborted.  A pipeline
// barrier only stalls when the role upstream of it stalls, so its bound is 4x the flag-wait
// bound: the wait at the root of a stall reports first.
static __device__ __noinline__ bool wait_bar_slow(const KParams& p, const SmemLayout& L,
                                                 uint32_t bar, uint32_t parity, uint32_t site) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*L.abort_flag) return false;
      if (globaltimer_ns() - t0 > 4 * p.timeout_ns) {
        raise_error(p, kDevTimeoutPipe, site, blockIdx.x, parity);
        *L.abort_flag = 1;
        return false;
      }
    }
  }
}
// The issuing threads wait once per k-block: the first test is inline (a call per wait costs
// the MMA issue loop about an eighth of its rate); the timed retry loop is out of line.
__device__ __forceinline__ bool wait_bar(const KParams& p, const SmemLayout& L, uint32_t bar,
                                        uint32_t parity, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(p, L, bar, parity, site);
}

// Bounded acquire-poll of a chunk's ready flag.
static __device__ __noinline__ bool wait_flag(const KParams& p, const SmemLayout& L, int32_t c) {
  const uint32_t* f = p.ready + c;
  unsigned long long* tr = p.trace;
  const int64_t tw = kTraceHead + 3 * static_cast<int64_t>(c);
  if (ld_acquire_gpu(f) == p.epoch) {
    trace_min(tr, tw + 2);
    return true;
  }
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(it < 64 ? 32 : 256);
    if (ld_acquire_gpu(f) == p.epoch) {
      if (tr != nullptr) {
        const uint64_t t1 = globaltimer_ns();
        atomicMin(tr + tw + 1, static_cast<unsigned long long>(t0));
        atomicMin(tr + tw + 2, static_cast<unsigned long long>(t1));
        atomicAdd(tr + 2, static_cast<unsigned long long>(t1 - t0));
        atomicAdd(tr + 3, 1ull);
      }
      return true;
    }
    if ((it & 7u) == 0u) {
      if (*L.abort_flag) return false;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        raise_error(p, kDevTimeoutFlag, static_cast<uint32_t>(c), blockIdx.x, p.epoch);
        *L.abort_flag = 1;
        return false;
      }
    }
  }
}

struct TileInfo {
  int32_t q, i, n, h;  // i: index of this CTA's 128-row m-tile
  int64_t row0, row_end, col0, col_end;
  bool valid;
};

// Clusters: the CL CTAs of a cluster work on the same tile of the order, each on its own 128 of
// the tile's CL * 128 rows, in cluster-rank order.  CTAs 2k and 2k+1 form a pair (tcgen05
// cta_group::2) whose even CTA issues the MMAs.
template <int CL>
__device__ __forceinline__ uint32_t cl_rank() {
  return CL > 1 ? (blockIdx.x % static_cast<uint32_t>(CL)) : 0u;
}

// Tile id at position pos of the order (identity in the baselines' plain launches); -1 past the
// end.  Each role fetches the next tile's id while it works on the current one, so the load's
// latency does not sit between two tiles.
__device__ __forceinline__ int32_t tile_id(const KParams& p, int32_t pos) {
  if (pos >= p.T) return -1;
  return p.plain ? pos : __ldg(p.order + pos);
}

template <int OP, int CL>
__device__ __forceinline__ TileInfo decode_tile(const KParams& p, int32_t t) {
  TileInfo ti;
  ti.valid = (t >= 0 && t < p.T);
  if (!ti.valid) t = 0;
  // an AllToAll baseline launch holds one destination block (Tnw column tiles) per rank
  const int32_t tn = (OP == kOpA2A && p.a2a_step >= 0) ? p.g.Tnw : p.g.Tn;
  const int32_t per_q = p.Tm * tn;
  ti.q = OP != kOpAG ? t / per_q : 0;
  const int32_t rem = t - ti.q * per_q;
  const int32_t it = rem / tn;
  ti.n = rem - it * tn;
  ti.i = CL * it + static_cast<int32_t>(cl_rank<CL>());
  ti.row0 = p.row_lo + static_cast<int64_t>(ti.i) * kBM;
  ti.row_end = min64(ti.row0 + kBM, p.row_hi);
  if (OP == kOpA2A) {
    int32_t c;
    if (p.a2a_step >= 0) {
      ti.h = (ti.q + p.a2a_step + 1) % p.g.W;
      c = ti.n;
    } else {
      ti.h = ti.n / p.g.Tnw;
      c = ti.n - ti.h * p.g.Tnw;
    }
    ti.col0 = static_cast<int64_t>(ti.h) * p.g.Nw + static_cast<int64_t>(c) * kBN;
    ti.col_end = static_cast<int64_t>(ti.h + 1) * p.g.Nw;
  } else {
    ti.h = 0;
    ti.col0 = static_cast<int64_t>(ti.n) * kBN;
    ti.col_end = p.g.N;
  }
  return ti;
}

// Compute CTAs are blockIdx.x >= copy_ctas; they (or their pairs) take the tile order one wave
// of pos_stride positions at a time (pos_at).
template <int CL>
__device__ __forceinline__ int32_t first_pos(const KParams& p) {
  return (static_cast<int32_t>(blockIdx.x) - p.copy_ctas) / CL;
}
template <int CL>
__device__ __forceinline__ int32_t pos_stride(const KParams& p) {
  return (static_cast<int32_t>(gridDim.x) - p.copy_ctas) / CL;
}
// The position a CTA (or pair) takes in wave k, the k-th run of pos_stride consecutive
// positions: slot (first_pos + k * rot) of the wave.  Every wave runs the same positions
// whatever rot is; with rot != 0 a CTA does not take the same slot in every wave, so tiles that
// cost more and recur at fixed slots (those cut by destination boundaries) spread over the CTAs.
// A position past the end (last wave) is skipped, not the end of the loop.
template <int CL>
__device__ __forceinline__ int32_t pos_at(const KParams& p, int32_t k) {
  const uint32_t S = static_cast<uint32_t>(pos_stride<CL>(p));
  const uint32_t r = static_cast<uint32_t>(p.rot) % S;
  const uint32_t slot = (static_cast<uint32_t>(first_pos<CL>(p)) + static_cast<uint32_t>(k) * r) % S;
  return k * static_cast<int32_t>(S) + static_cast<int32_t>(slot);
}
template <int CL>
__device__ __forceinline__ int32_t wave_count(const KParams& p) {
  const int32_t S = pos_stride<CL>(p);
  return (p.T + S - 1) / S;
}

// Warp-wide bounded wait: every lane polls, a vote makes the outcome the warp's, so all lanes
// leave a loop together (the producer and MMA roles run as whole warps that stay converged;
// one elected lane issues the TMA loads or MMAs).
__device__ __forceinline__ bool warp_wait_bar(const KParams& p, const SmemLayout& L, uint32_t bar,
                                             uint32_t parity, uint32_t site) {
  return __all_sync(0xffffffffu, wait_bar(p, L, bar, parity, site));
}

// ============================================================================ producer
template <int OP, int CL, int NS>
__device__ void run_producer(const KParams& p, const SmemLayout& L) {
  constexpr bool PAIR = CL > 1;
  constexpr int NB = b_slabs(PAIR);
  // a pair's loads complete on its even CTA's barriers; that CTA expects both CTAs' bytes
  const uint32_t rank = cl_rank<CL>();
  const bool leader = (rank & 1u) == 0u;
  // stage s: barriers 8 s bytes after stage 0's, buffers s stages after stage 0's
  const uint32_t full0 = L.full(0), empty0 = L.empty(0);
  const uint32_t a_smem0 = smem_u32(L.a), b_smem0 = smem_u32(L.b);
  const bool b_keep = OP == kOpRS && (p.l2_hints & 2) != 0;
  const uint64_t pol_b = l2_policy_evict_last();
  uint32_t full0_lead = full0;  // stage 0's full barrier in the pair leader (cluster address)
  if constexpr (PAIR) full0_lead = mapa_shared(full0, rank & ~1u);
  uint32_t kit = 0;  // k-blocks issued so far (the last one, if any, is kit - 1)
  const int32_t nwaves = wave_count<CL>(p);
  int32_t t_next = tile_id(p, pos_at<CL>(p, 0));
  for (int32_t k = 0; k < nwaves; ++k) {
    const int32_t pos = pos_at<CL>(p, k);
    const int32_t t_cur = t_next;
    t_next = tile_id(p, pos_at<CL>(p, k + 1));
    if (pos >= p.T) continue;
    const TileInfo ti = decode_tile<OP, CL>(p, t_cur);
    if (!ti.valid) {
      if (elect_one()) raise_error(p, kDevBadTile, static_cast<uint32_t>(pos), blockIdx.x, 0);
      __syncwarp();
      continue;
    }
    // local HBM as the cache of remote memory: the own rank's rows need no transfer
    const int64_t own0 = static_cast<int64_t>(p.g.rank) * p.g.Ms;
    const bool own_tile =
        OP == kOpAG && p.own_in_place && ti.row0 >= own0 && ti.row_end <= own0 + p.g.Ms;
    if (OP == kOpAG && p.wait_flags && !own_tile) {
      // consumer_tile_wait: every chunk holding one of this tile's rows must have landed
      // (polled by the lane that issues the loads)
      bool ok = true;
      if (elect_one()) {
        for (int64_t g = ti.row0; g < ti.row_end && ok;) {
          int32_t s, j;
          row_chunk(p.g, g, s, j);
          const int32_t c = s * p.g.nC + j;
          const bool cached =
              c < kReadyBitsWords * 32 && ((L.ready_bits[c >> 5] >> (c & 31)) & 1u);
          if (!cached) {
            ok = wait_flag(p, L, c);
            if (ok && c < kReadyBitsWords * 32) L.ready_bits[c >> 5] |= 1u << (c & 31);
          }
          g = static_cast<int64_t>(s) * p.g.Ms +
              min64(static_cast<int64_t>(j + 1) * p.g.Cr, p.g.Ms);
        }
        // the rows were written by other agents through the generic proxy (or the copy
        // engine); the TMA loads below read through the async proxy
        if (ok) fence_proxy_async_global();
      }
      if (__any_sync(0xffffffffu, !ok)) break;
    }
    const CUtensorMap* tA = &p.tmA[OP != kOpAG ? ti.q : (own_tile ? 1 : 0)];
    const CUtensorMap* tB = &p.tmB[OP != kOpAG ? ti.q : 0];
    int32_t a_row = static_cast<int32_t>(own_tile ? ti.row0 - own0 : ti.row0);
    if (OP == kOpAG && p.a_from_shards) {
      // co-located pull: this CTA's 128 rows lie in one shard ((M/W) % 128 == 0); the loads
      // complete on the stage's mbarrier like any operand load
      const int32_t s = static_cast<int32_t>(ti.row0 / p.g.Ms);
      tA = &p.tmA[s];
      a_row = static_cast<int32_t>(ti.row0 - static_cast<int64_t>(s) * p.g.Ms);
    }
    // this CTA's columns of B: all 256, or its half of the pair's
    const int32_t b_col = static_cast<int32_t>(ti.col0) + static_cast<int32_t>(rank & 1u) * (NB * 64);
    bool ok = true;
    for (int32_t kb = 0; kb < p.KB; ++kb, ++kit) {
      const int st = static_cast<int>(kit % NS);
      const uint32_t ph = (kit / NS) & 1u;
      const uint32_t sst = static_cast<uint32_t>(st);
      if (!warp_wait_bar(p, L, empty0 + 8u * sst, ph ^ 1u, 100 + st)) { ok = false; break; }
      if (elect_one()) {
        const uint32_t a_dst = a_smem0 + sst * kAStage;
        const uint32_t b_dst = b_smem0 + sst * b_stage_bytes(PAIR);
        const uint32_t fb = full0 + 8u * sst;
        if constexpr (PAIR) {
          const uint32_t bar = full0_lead + 8u * sst;
          if (leader) mbar_expect_tx(fb, 2 * (kAStage + b_stage_bytes(PAIR)));
          tma_load_2d_pair(a_dst, tA, kb * kBK, a_row, bar);
          if (b_keep) {
#pragma unroll
            for (int jj = 0; jj < NB; ++jj)
              tma_load_2d_pair_hint(b_dst + jj * kBSlab, tB, b_col + jj * 64, kb * kBK, bar, pol_b);
          } else {
#pragma unroll
            for (int jj = 0; jj < NB; ++jj)
              tma_load_2d_pair(b_dst + jj * kBSlab, tB, b_col + jj * 64, kb * kBK, bar);
          }
        } else {
          mbar_expect_tx(fb, kAStage + b_stage_bytes(PAIR));
          tma_load_2d(a_dst, tA, kb * kBK, a_row, fb);
          if (b_keep) {
#pragma unroll
            for (int jj = 0; jj < NB; ++jj)
              tma_load_2d_hint(b_dst + jj * kBSlab, tB, b_col + jj * 64, kb * kBK, fb, pol_b);
          } else {
#pragma unroll
            for (int jj = 0; jj < NB; ++jj)
              tma_load_2d(b_dst + jj * kBSlab, tB, b_col + jj * 64, kb * kBK, fb);
          }
        }
      }
      __syncwarp();
    }
    if (!ok) break;
  }
  if (__any_sync(0xffffffffu, *L.abort_flag != 0) && leader) {
    // let every TMA load issued into this stage ring land before the CTA can exit (a pair's
    // leader barrier counts the other CTA's bytes as well)
    // the last k-block issued into stage s is the largest k < kit with k % NS == s
    for (int s = 0; s < NS; ++s) {
      if (kit <= static_cast<uint32_t>(s)) continue;
      const uint32_t last = (kit - 1u) - ((kit - 1u - static_cast<uint32_t>(s)) % NS);
      const uint32_t ph = (last / NS) & 1u;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(L.full(s), ph) && globaltimer_ns() - t0 < p.timeout_ns) {
      }
    }
  }
}

// ============================================================================ MMA issuer
// The whole MMA warp runs the loop, so it stays converged, and one elected lane issues the
// MMAs and commits: issued by a lone lane of a diverged warp, CTA-pair MMAs (M = 256, N = 256,
// K = 16) go out every 135 clocks instead of every 128.

template <int OP, int CL, int NS>
__device__ void run_mma(const KParams& p, const SmemLayout& L, uint32_t tmem_base) {
  constexpr bool PAIR = CL > 1;
  // commit masks: a stage and an accumulator belong to both CTAs of the pair
  const uint32_t rank = cl_rank<CL>();
  const uint16_t stage_mask = 0x3;
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (rank & ~1u));
  // a pair's MMA has M = 256: rows 0-127 from the even CTA, 128-255 from the odd one
  constexpr uint32_t kIdesc = idesc_bf16_f32(PAIR ? 2 * kBM : kBM, kBN, /*B MN-major*/ 1);
  uint32_t kit = 0;
  int32_t tl = 0;
  bool issued = false;
  // what the k-loop touches, in registers: stage s's barriers are 8 s bytes after stage 0's,
  // its descriptors (s * stage bytes) >> 4 after stage 0's (the start-address field, which
  // cannot carry: shared addresses stay below 256 KB)
  const uint32_t full0 = L.full(0), empty0 = L.empty(0);
  const uint64_t adesc0 = smem_desc_sw128(smem_u32(L.a), 16, 1024);
  const uint64_t bdesc0 = smem_desc_sw128(smem_u32(L.b), kBSlab, 1024);
  const int32_t nwaves = wave_count<CL>(p);
  int32_t t_next = tile_id(p, pos_at<CL>(p, 0));
  for (int32_t k = 0; k < nwaves; ++k) {
    const int32_t pos = pos_at<CL>(p, k);
    const int32_t t_cur = t_next;
    t_next = tile_id(p, pos_at<CL>(p, k + 1));
    if (pos >= p.T) continue;
    const TileInfo ti = decode_tile<OP, CL>(p, t_cur);
    if (!ti.valid) continue;
    const int acc = tl & 1;
    const uint32_t aph = (static_cast<uint32_t>(tl) >> 1) & 1u;
    if (!warp_wait_bar(p, L, L.tempty(acc), aph ^ 1u, 200 + acc)) break;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
    bool ok = true;
    for (int32_t kb = 0; kb < p.KB; ++kb, ++kit) {
      const int st = static_cast<int>(kit % NS);
      const uint32_t ph = (kit / NS) & 1u;
      // the stage was filled by TMA (async proxy) and is read by the MMAs (async proxy): the
      // barrier's completion orders them; no tcgen05 fence here, which would hold the issue
      // of this k-block until the MMAs in flight have finished
      const uint32_t fb = full0 + 8u * static_cast<uint32_t>(st);
      if (!warp_wait_bar(p, L, fb, ph, 300 + st)) { ok = false; break; }
      const uint64_t ad0 =
          adesc0 + static_cast<uint64_t>((static_cast<uint32_t>(st) * kAStage) >> 4);
      const uint64_t bd0 =
          bdesc0 + static_cast<uint64_t>((static_cast<uint32_t>(st) * b_stage_bytes(PAIR)) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // A: K-major rows of 128 B, 8-row groups 1024 B apart (SBO); +32 B per 16 k
          const uint64_t ad = ad0 + static_cast<uint64_t>(kk * (32 >> 4));
          // B: MN-major; 64-column slabs 8 KB apart (LBO), 8 k-row groups 1 KB apart (SBO);
          // +2 KB per 16 k
          const uint64_t bd = bd0 + static_cast<uint64_t>(kk * (2048 >> 4));
          if constexpr (PAIR)
            umma_bf16_pair(d_tmem, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
          else
            umma_bf16(d_tmem, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
        }
        // frees the stage (in both CTAs of a pair) once these MMAs have read it
        const uint32_t eb = empty0 + 8u * static_cast<uint32_t>(st);
        if constexpr (PAIR) umma_commit_pair(eb, stage_mask); else umma_commit(eb);
      }
      __syncwarp();
      issued = true;
    }
    if (!ok) break;
    // accumulator ready for the epilogue (of both CTAs)
    if (elect_one()) {
      if constexpr (PAIR) umma_commit_pair(L.tfull(acc), pair_mask); else umma_commit(L.tfull(acc));
    }
    __syncwarp();
    ++tl;
  }
  if (__any_sync(0xffffffffu, *L.abort_flag != 0) && issued) {
    if (elect_one()) {
      if constexpr (PAIR) umma_commit_pair(L.fin(), static_cast<uint16_t>(1u << rank));
      else umma_commit(L.fin());
    }
    __syncwarp();
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(L.fin(), 0) && globaltimer_ns() - t0 < p.timeout_ns) {
    }
  }
}

// ============================================================================ epilogue
// Activation of the fp32 accumulator before it is stored (the first GEMM of a feed-forward
// block): GELU in its tanh form, 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), or SiLU,
// x / (1 + exp(-x)); CUDA's tanhf / expf.
__device__ __forceinline__ void apply_activation(uint32_t (&v)[32], int act) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float x = __uint_as_float(v[e]);
    float y;
    if (act == 1)
      y = 0.5f * x * (1.0f + tanhf(0.7978845608028654f * (x + 0.044715f * x * x * x)));
    else
      y = x / (1.0f + expf(-x));
    v[e] = __float_as_uint(y);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <bool F32>
__device__ __forceinline__ void store_row32(void* out, int64_t ldc, int64_t row, int64_t c0,
                                            int64_t N, const uint32_t (&v)[32]) {
  if (F32) {
    float* dst = reinterpret_cast<float*>(out) + row * ldc + c0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (c0 + u * 8 < N) {
        reinterpret_cast<float4*>(dst + u * 8)[0] =
            make_float4(__uint_as_float(v[u * 8 + 0]), __uint_as_float(v[u * 8 + 1]),
                        __uint_as_float(v[u * 8 + 2]), __uint_as_float(v[u * 8 + 3]));
        reinterpret_cast<float4*>(dst + u * 8)[1] =
            make_float4(__uint_as_float(v[u * 8 + 4]), __uint_as_float(v[u * 8 + 5]),
                        __uint_as_float(v[u * 8 + 6]), __uint_as_float(v[u * 8 + 7]));
      }
    }
  } else {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(out) + row * ldc + c0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (c0 + u * 8 < N) {
        uint4 w;
        w.x = pack_bf16x2(v[u * 8 + 0], v[u * 8 + 1]);
        w.y = pack_bf16x2(v[u * 8 + 2], v[u * 8 + 3]);
        w.z = pack_bf16x2(v[u * 8 + 4], v[u * 8 + 5]);
        w.w = pack_bf16x2(v[u * 8 + 6], v[u * 8 + 7]);
        *reinterpret_cast<uint4*>(dst) = w;
      }
      dst += 8;
    }
  }
}

__device__ __forceinline__ float4 ldcg_f4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// ---------------------------------------------------------------------------- RS folding
// A ReduceScatter unit is (the rows of m-tile i inside one chunk of destination s) x column
// tile n.  Its W partials are summed in the fixed source order d = q = 0..W-1: the order in
// which the schedule produces them (the virtual ranks run one after another, each in its own
// scatter order).  The running fp32 sum S_d = S_{d-1} + P_d lives in `acc` ([M][N], global
// rows); S_{W-1} is rounded once into out_s.  A partial that is
// ready before its predecessors are folded waits in park slot (s, d).  One 32-bit word per unit
// holds the number of partials folded so far (bits 0-7) and which ones are parked (bit 8+d);
// whoever moves the count to d, or parks d after the count reached d, folds d: exactly one
// tile does, and nobody waits.
__device__ __forceinline__ int32_t fold_index(int32_t s, int32_t q, int32_t W) {
  (void)s;
  (void)W;
  return q;
}
__device__ __forceinline__ float* acc_ptr(const KParams& p, int64_t row, int64_t col) {
  return p.recv + row * p.g.N + col;
}
__device__ __forceinline__ float* park_ptr(const KParams& p, int32_t s, int32_t d, int64_t lr,
                                           int64_t col) {
  const size_t slot = static_cast<size_t>(s) * (p.g.W - 1) + (d - 1);  // d = 0 never parks
  return p.recv + static_cast<size_t>(p.g.M) * p.g.N +
         (slot * p.g.Ms + lr) * static_cast<size_t>(p.g.N) + col;
}

// Final result of 8 columns of row lr of destination s: into out_s (ReduceScatter), or at
// global row s*Ms + lr into every rank's output (AllReduce).
template <bool F32>
__device__ __forceinline__ void store_out8(const KParams& p, int32_t s, int64_t lr, int64_t col,
                                           const float (&a)[8]) {
  const int ncopy = p.ar_copies > 0 ? p.ar_copies : 1;
  const int64_t row = p.ar_copies > 0 ? static_cast<int64_t>(s) * p.g.Ms + lr : lr;
  uint4 w;
  if (!F32) {
    w.x = pack_bf16x2(__float_as_uint(a[0]), __float_as_uint(a[1]));
    w.y = pack_bf16x2(__float_as_uint(a[2]), __float_as_uint(a[3]));
    w.z = pack_bf16x2(__float_as_uint(a[4]), __float_as_uint(a[5]));
    w.w = pack_bf16x2(__float_as_uint(a[6]), __float_as_uint(a[7]));
  }
  for (int r = 0; r < ncopy; ++r) {
    void* out = p.out[p.ar_copies > 0 ? r : s];
    if (F32) {
      float* dst = reinterpret_cast<float*>(out) + row * p.ldc + col;
      reinterpret_cast<float4*>(dst)[0] = make_float4(a[0], a[1], a[2], a[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(a[4], a[5], a[6], a[7]);
    } else {
      *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + row * p.ldc + col) = w;
    }
  }
}
template <bool F32>
__device__ __forceinline__ void store_out4(const KParams& p, int32_t s, int64_t lr, int64_t col,
                                           const float4& r4) {
  const int ncopy = p.ar_copies > 0 ? p.ar_copies : 1;
  const int64_t row = p.ar_copies > 0 ? static_cast<int64_t>(s) * p.g.Ms + lr : lr;
  for (int r = 0; r < ncopy; ++r) {
    void* out = p.out[p.ar_copies > 0 ? r : s];
    if (F32) {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + row * p.ldc + col) = r4;
    } else {
      uint2 w;
      w.x = pack_bf16x2(__float_as_uint(r4.x), __float_as_uint(r4.y));
      w.y = pack_bf16x2(__float_as_uint(r4.z), __float_as_uint(r4.w));
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + row * p.ldc + col) = w;
    }
  }
}

// One thread, one row, 32 columns: fold this tile's partial (index d, in registers) into the
// running sum; the last fold writes out_s.
template <bool F32>
__device__ __forceinline__ void fold_row32(const KParams& p, int32_t s, int64_t row, int64_t lr,
                                           int32_t d, int64_t c0, const uint32_t (&v)[32]) {
  float* acc = acc_ptr(p, row, c0);
  float4 x[8];
  if (d > 0) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (c0 + u * 4 < p.g.N) x[u] = ldcg_f4(acc + u * 4);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    if (c0 + u * 8 >= p.g.N) break;
    float a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = __uint_as_float(v[u * 8 + e]);
    if (d > 0) {
      a[0] = x[2 * u].x + a[0]; a[1] = x[2 * u].y + a[1];
      a[2] = x[2 * u].z + a[2]; a[3] = x[2 * u].w + a[3];
      a[4] = x[2 * u + 1].x + a[4]; a[5] = x[2 * u + 1].y + a[5];
      a[6] = x[2 * u + 1].z + a[6]; a[7] = x[2 * u + 1].w + a[7];
    }
    if (d == p.g.W - 1) {
      store_out8<F32>(p, s, lr, c0 + u * 8, a);
    } else {
      reinterpret_cast<float4*>(acc + u * 8)[0] = make_float4(a[0], a[1], a[2], a[3]);
      reinterpret_cast<float4*>(acc + u * 8)[1] = make_float4(a[4], a[5], a[6], a[7]);
    }
  }
}

// The 128 epilogue threads fold parked partial e of rows [lo, hi) (destination s), column tile n.
// Each thread has kParkVecs vectors of the running sum and of the parked partial in flight at
// once (a unit is up to 128 x 256 fp32: 64 vectors per thread, which one at a time would be
// 64 dependent round trips to memory).
constexpr int kParkVecs = 8;
template <bool F32>
__device__ void fold_parked(const KParams& p, int32_t s, int64_t lo, int64_t hi, int32_t n,
                            int32_t e, int et) {
  const int64_t c0 = static_cast<int64_t>(n) * kBN;
  const int32_t nv = static_cast<int32_t>(min64(kBN, p.g.N - c0)) >> 2;
  const int32_t nrows = static_cast<int32_t>(hi - lo);
  const int32_t total = nrows * nv;
  for (int32_t base = et; base < total; base += 128 * kParkVecs) {
    float4 a[kParkVecs], b[kParkVecs];
#pragma unroll
    for (int u = 0; u < kParkVecs; ++u) {
      const int32_t idx = base + u * 128;
      if (idx < total) {
        const int32_t r = idx / nv;
        const int64_t row = lo + r;
        const int64_t col = c0 + (idx - r * nv) * 4;
        a[u] = ldcg_f4(acc_ptr(p, row, col));
        b[u] = ldcg_f4(park_ptr(p, s, e, row - static_cast<int64_t>(s) * p.g.Ms, col));
      }
    }
#pragma unroll
    for (int u = 0; u < kParkVecs; ++u) {
      const int32_t idx = base + u * 128;
      if (idx < total) {
        const int32_t r = idx / nv;
        const int64_t row = lo + r;
        const int64_t lr = row - static_cast<int64_t>(s) * p.g.Ms;
        const int64_t col = c0 + (idx - r * nv) * 4;
        const float4 r4 = make_float4(a[u].x + b[u].x, a[u].y + b[u].y, a[u].z + b[u].z,
                                      a[u].w + b[u].w);
        if (e == p.g.W - 1) {
          store_out4<F32>(p, s, lr, col, r4);
        } else {
          *reinterpret_cast<float4*>(acc_ptr(p, row, col)) = r4;
        }
      }
    }
  }
}

// Fold parked partials e, e+1, ... of one unit while they are there (all 128 epilogue threads).
template <bool F32>
__device__ void fold_chain(const KParams& p, const SmemLayout& L, int32_t s, int64_t lo,
                           int64_t hi, int32_t n, int32_t e, uint32_t* word, int et) {
  for (;;) {
    __threadfence();
    fold_parked<F32>(p, s, lo, hi, n, e, et);
    __threadfence();
    named_bar_sync(1, 128);
    if (et == 0) {
      int next = -1;
      if (e == p.g.W - 1) {
        *word = 0u;  // all W folded: ready for the next call
      } else {
        // count one more folded, clear e's parked bit; is e+1 parked already?
        const uint32_t old = atom_add_acq_rel_gpu(word, 1u - (1u << (8 + e)));
        if ((old >> (8 + e + 1)) & 1u) next = e + 1;
      }
      *L.unit_flag = next;
    }
    named_bar_sync(1, 128);
    const int next = *L.unit_flag;
    named_bar_sync(1, 128);
    if (next < 0) break;
    e = next;
  }
}

template <int OP, bool F32, int CL>
__device__ void run_epilogue(const KParams& p, const SmemLayout& L, uint32_t tmem_base,
                             int warp, int lane, bool staging_free) {
  constexpr bool PAIR = CL > 1;
  constexpr bool RS = OP == kOpRS;
  constexpr bool A2A = OP == kOpA2A;
  constexpr bool kStoreF32 = RS || F32;  // ReduceScatter partials are fp32
  // AllGather: C's 32-column boxes go out as TMA stores from the staging buffers (which the
  // co-located TMA transfer, when there is one, needs for itself)
  const bool c_tma =
      (OP == kOpAG || (A2A && !p.plain)) && p.c_tma != 0 && staging_free;
  const int qd = warp - 4;  // TMEM lane quadrant this warp may read
  const int et = threadIdx.x - 128;
  const bool fused_rs = RS && !p.plain;
  const bool fused_a2a = A2A && !p.plain;
  int32_t tl = 0;
  const bool stream_sums = RS && (p.l2_hints & 1) != 0;  // running sums pass through L2 once
  const uint64_t pol_s = l2_policy_evict_first();
  uint32_t stage_ctr = 0;           // running-sum staging buffer in use (alternates)
  uint32_t ld_par[2] = {0u, 0u};    // phase of each staging buffer's load barrier
  // a pair's accumulator is released on the even CTA's barrier, by the warps of both CTAs
  uint32_t tempty_bar0 = L.tempty(0), tempty_bar1 = L.tempty(1);
  if constexpr (PAIR) {
    const uint32_t lead = cl_rank<CL>() & ~1u;
    tempty_bar0 = mapa_shared(tempty_bar0, lead);
    tempty_bar1 = mapa_shared(tempty_bar1, lead);
  }
  const int32_t nwaves = wave_count<CL>(p);
  int32_t t_next = tile_id(p, pos_at<CL>(p, 0));
  for (int32_t k = 0; k < nwaves; ++k) {
    const int32_t pos = pos_at<CL>(p, k);
    const int32_t t_cur = t_next;
    t_next = tile_id(p, pos_at<CL>(p, k + 1));
    if (pos >= p.T) continue;
    const TileInfo ti = decode_tile<OP, CL>(p, t_cur);
    if (!ti.valid) continue;
    const int acc = tl & 1;
    const uint32_t ph = (static_cast<uint32_t>(tl) >> 1) & 1u;
    int ok = 1;
    if (lane == 0) ok = wait_bar(p, L, L.tfull(acc), ph, 400 + acc) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (fused_rs || fused_a2a) {
      // all four epilogue warps agree before they meet at the named barriers below
      if (lane == 0) L.vote[(tl & 1) * 4 + qd] = ok;
      named_bar_sync(1, 128);
      ok = L.vote[(tl & 1) * 4 + 0] & L.vote[(tl & 1) * 4 + 1] & L.vote[(tl & 1) * 4 + 2] &
           L.vote[(tl & 1) * 4 + 3];
    }
    if (!ok) break;
    tc_fence_after();
    const int64_t row = ti.row0 + qd * 32 + lane;
    const bool row_ok = row < ti.row_end;
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) +
                           static_cast<uint32_t>(acc * kBN);
    // ReduceScatter: the tile's rows split at chunk boundaries into units ("pieces"); find
    // which of them this tile folds in order (all earlier partials folded already)
    int32_t c_first = 0;
    uint32_t* words = nullptr;
    if (fused_rs) {
      int32_t s0, j0;
      row_chunk(p.g, ti.row0, s0, j0);
      c_first = s0 * p.g.nC + j0;
      words = p.unit_cnt +
              (static_cast<int64_t>(ti.i) * p.g.Tn + ti.n) * static_cast<int64_t>(p.pieces_max);
      if (et == 0) {
        uint32_t m[4] = {0u, 0u, 0u, 0u};
        int k = 0;
        for (int64_t g = ti.row0; g < ti.row_end; ++k) {
          int32_t s, j;
          row_chunk(p.g, g, s, j);
          const uint32_t st = ld_acquire_gpu(words + k);
          if (static_cast<int32_t>(st & 0xffu) == fold_index(s, ti.q, p.g.W))
            m[k >> 5] |= 1u << (k & 31);
          g = static_cast<int64_t>(s) * p.g.Ms + min64(static_cast<int64_t>(j + 1) * p.g.Cr, p.g.Ms);
        }
        for (int w = 0; w < 4; ++w) L.last_mask[w] = m[w];
      }
      named_bar_sync(1, 128);
      __threadfence();
    }
    int32_t s_row = 0, j_row = 0, d_row = 0;
    bool in_order = false;
    int64_t lr = 0;
    if (RS && row_ok) {
      row_chunk(p.g, row, s_row, j_row);
      lr = row - static_cast<int64_t>(s_row) * p.g.Ms;
      d_row = fold_index(s_row, ti.q, p.g.W);
      if (fused_rs) {
        const int32_t k = s_row * p.g.nC + j_row - c_first;
        in_order = (L.last_mask[k >> 5] >> (k & 31)) & 1u;
      }
    }
    // Tiles move their running sums with TMA in 128 x 32 fp32 boxes through a 128-byte-swizzled
    // staging buffer: the first source stores its partial, a middle one reduce-adds it into the
    // running sum, the last one loads the running sum, adds and stores the final sums (a park
    // slot takes a partial that is early).  A whole 128-row tile inside one unit always can (in
    // order or parked); a tile cut by chunk or destination boundaries, or the ragged last tile,
    // can when every piece folds in order (the running sums are one [M][N] array, so the box
    // spans the pieces) and, for the last partial of a ReduceScatter tile, its rows lie in at
    // most two destinations (the second's rows are stored from registers).  The rest go row by
    // row.
    bool tma_tile = false;
    int32_t t_s = 0, t_s1 = 0, t_d = 0;
    int64_t t_lr0 = 0;
    bool t_in_order = false;
    if (fused_rs && ti.row_end > ti.row0) {
      int32_t s0, j0, s1, j1;
      row_chunk(p.g, ti.row0, s0, j0);
      row_chunk(p.g, ti.row_end - 1, s1, j1);
      const int32_t d = fold_index(s0, ti.q, p.g.W);  // every piece's: sources fold in order
      if (s0 == s1 && j0 == j1 && ti.row_end - ti.row0 == kBM) {
        tma_tile = true;
        t_in_order = L.last_mask[0] & 1u;
      } else {
        const int32_t np = (s1 * p.g.nC + j1) - (s0 * p.g.nC + j0) + 1;  // pieces of the tile
        bool all = true;
        for (int32_t k = 0; k < np && all; ++k) all = (L.last_mask[k >> 5] >> (k & 31)) & 1u;
        if (all && (d < p.g.W - 1 || p.ar_copies > 0 || s1 <= s0 + 1)) {
          tma_tile = true;
          t_in_order = true;
        }
      }
      if (tma_tile) {
        t_s = s0;
        t_s1 = s1;
        t_d = d;
        t_lr0 = ti.row0 - static_cast<int64_t>(s0) * p.g.Ms;
      }
    }
    if (tma_tile) {
      // a middle source adds its partial into the running sum in place (TMA reduce-add: the
      // fp32 add of the loading path, done by the memory system, so nothing waits for a load);
      // the first one stores it, the last one loads the running sum to round the final sum
      const bool red = t_in_order && t_d > 0 && t_d < p.g.W - 1 && p.rs_reduce != 0;
      const bool load = t_in_order && t_d > 0 && !red;
      const bool last = t_in_order && t_d == p.g.W - 1;
      const CUtensorMap* store_map = t_in_order ? &p.tmAcc : &p.tmPark;
      const int32_t store_y =
          t_in_order ? static_cast<int32_t>(ti.row0)
                     : static_cast<int32_t>((static_cast<int64_t>(t_s) * (p.g.W - 1) + t_d - 1) *
                                                p.g.Ms + t_lr0);
      const int r = qd * 32 + lane;  // this thread's row of the tile
      const int ncb = static_cast<int>(min64(kBN, p.g.N - ti.col0) + 31) / 32;  // 32-column boxes
      // the final sums of a ReduceScatter tile across two destinations: the box goes to the
      // first one as a TMA store (its tensor map ends at that destination's last row), and the
      // threads whose rows belong to the second store them from registers
      const int64_t split_row = static_cast<int64_t>(t_s + 1) * p.g.Ms;
      const bool row_to_s1 = last && p.ar_copies == 0 && t_s1 != t_s && ti.row0 + r >= split_row &&
                             ti.row0 + r < ti.row_end;
      const int64_t lr1 = row_to_s1 ? ti.row0 + r - split_row : 0;
      // Box cb+1's running sum is loaded into the other buffer while box cb is processed.  The
      // buffers are free at the start of a tile (its predecessor waited for all its stores).
      if (et == 0 && red) fence_proxy_async_global();  // as below, for the reductions
      if (et == 0 && load) {
        // the unit's word was acquired through the generic proxy; the loads below are TMA
        fence_proxy_async_global();
        const int b0 = static_cast<int>(stage_ctr & 1u);
        mbar_expect_tx(L.copyb(b0), kCopyBuf);
        if (stream_sums)
          tma_load_2d_hint(smem_u32(L.copy + b0 * kCopyBuf), &p.tmAcc, static_cast<int32_t>(ti.col0),
                           static_cast<int32_t>(ti.row0), L.copyb(b0), pol_s);
        else
          tma_load_2d(smem_u32(L.copy + b0 * kCopyBuf), &p.tmAcc, static_cast<int32_t>(ti.col0),
                      static_cast<int32_t>(ti.row0), L.copyb(b0));
      }
#pragma unroll 1
      for (int cb = 0; cb < ncb; ++cb) {
        const int64_t c0 = ti.col0 + cb * 32;
        const int b = static_cast<int>(stage_ctr & 1u);
        uint8_t* buf = L.copy + b * kCopyBuf;
        if (et == 0 && red) {
          bulk_wait_read<1>();  // box cb-2's reduction has read this buffer
        } else if (et == 0) {
          bulk_wait_read<0>();  // box cb-1's store has read the other buffer
          if (load && cb + 1 < ncb) {
            mbar_expect_tx(L.copyb(b ^ 1), kCopyBuf);
            if (stream_sums)
              tma_load_2d_hint(smem_u32(L.copy + (b ^ 1) * kCopyBuf), &p.tmAcc,
                               static_cast<int32_t>(c0 + 32), static_cast<int32_t>(ti.row0),
                               L.copyb(b ^ 1), pol_s);
            else
              tma_load_2d(smem_u32(L.copy + (b ^ 1) * kCopyBuf), &p.tmAcc,
                          static_cast<int32_t>(c0 + 32), static_cast<int32_t>(ti.row0),
                          L.copyb(b ^ 1));
          }
        }
        named_bar_sync(1, 128);
        uint32_t v[32];
        tmem_ld32(tbase + cb * 32, v);
        if (load) {
          wait_bar(p, L, L.copyb(b), ld_par[b], 600 + b);
          ld_par[b] ^= 1u;
        }
        float4* rowp = reinterpret_cast<float4*>(buf + r * 128);
        float a[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) a[e] = __uint_as_float(v[e]);
        if (load) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 x = rowp[c ^ (r & 7)];
            a[4 * c + 0] = x.x + a[4 * c + 0];
            a[4 * c + 1] = x.y + a[4 * c + 1];
            a[4 * c + 2] = x.z + a[4 * c + 2];
            a[4 * c + 3] = x.w + a[4 * c + 3];
          }
        }
        if (last && !F32) {
          // the final sum, rounded to bf16, as dense 64-byte rows of the box once every thread
          // has read its running-sum row out of the same buffer
          named_bar_sync(1, 128);
          uint4* orow = reinterpret_cast<uint4*>(buf + r * 64);
          __nv_bfloat16* orow1 = reinterpret_cast<__nv_bfloat16*>(p.out[t_s1]) + lr1 * p.ldc + c0;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(__float_as_uint(a[8 * u + 0]), __float_as_uint(a[8 * u + 1]));
            w.y = pack_bf16x2(__float_as_uint(a[8 * u + 2]), __float_as_uint(a[8 * u + 3]));
            w.z = pack_bf16x2(__float_as_uint(a[8 * u + 4]), __float_as_uint(a[8 * u + 5]));
            w.w = pack_bf16x2(__float_as_uint(a[8 * u + 6]), __float_as_uint(a[8 * u + 7]));
            orow[u] = w;
            if (row_to_s1 && c0 + u * 8 < p.g.N) reinterpret_cast<uint4*>(orow1)[u] = w;
          }
        } else {
          // the running sum (or the fp32 final sum) in the box's swizzled layout
#pragma unroll
          for (int c = 0; c < 8; ++c)
            rowp[c ^ (r & 7)] = make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
          if (row_to_s1) {  // fp32 final sums of the second destination's rows
            float* orow1 = reinterpret_cast<float*>(p.out[t_s1]) + lr1 * p.ldc + c0;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              if (c0 + c * 4 < p.g.N)
                reinterpret_cast<float4*>(orow1)[c] =
                    make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (et == 0) {
          if (red) {
            if (stream_sums)
              tma_reduce_add_2d_hint(&p.tmAcc, smem_u32(buf), static_cast<int32_t>(c0), store_y,
                                     pol_s);
            else
              tma_reduce_add_2d(&p.tmAcc, smem_u32(buf), static_cast<int32_t>(c0), store_y);
          } else if (!last) {
            if (stream_sums)
              tma_store_2d_hint(store_map, smem_u32(buf), static_cast<int32_t>(c0), store_y, pol_s);
            else
              tma_store_2d(store_map, smem_u32(buf), static_cast<int32_t>(c0), store_y);
          } else {
            // one TMA store per output: out_s (ReduceScatter), every rank's copy (AllReduce)
            const int ncopy = p.ar_copies > 0 ? p.ar_copies : 1;
            const int32_t oy = static_cast<int32_t>(p.ar_copies > 0 ? ti.row0 : t_lr0);
            for (int cp = 0; cp < ncopy; ++cp) {
              const CUtensorMap* om = &p.tmOut[p.ar_copies > 0 ? cp : t_s];
              if (stream_sums)
                tma_store_2d_hint(om, smem_u32(buf), static_cast<int32_t>(c0), oy, pol_s);
              else
                tma_store_2d(om, smem_u32(buf), static_cast<int32_t>(c0), oy);
            }
          }
          bulk_commit();
        }
        ++stage_ctr;
      }
      if (et == 0) {
        bulk_wait<0>();  // the running sum (or parked partial) is in global memory
        fence_proxy_async_global();
      }
    }
    if (c_tma) {
      // Each thread writes its row of the box into a staging buffer (bf16: dense 64-byte rows;
      // fp32: 128-byte rows in the 128-byte swizzle), then one thread stores the box; the
      // tensor map clips rows at M and columns at N.  A buffer is rewritten once the store
      // issued from it two boxes earlier has read it.
      const int r = qd * 32 + lane;
      const int ncb = static_cast<int>(min64(kBN, ti.col_end - ti.col0) + 31) / 32;
#pragma unroll 1
      for (int cb = 0; cb < ncb; ++cb) {
        uint8_t* buf = L.copy + (stage_ctr & 1u) * kCopyBuf;
        uint32_t v[32];
        tmem_ld32(tbase + cb * 32, v);
        if (p.act) apply_activation(v, p.act);
        if (et == 0) bulk_wait_read<1>();
        named_bar_sync(1, 128);
        if (F32) {
          float4* rowp = reinterpret_cast<float4*>(buf + r * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            rowp[c ^ (r & 7)] = make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                            __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
        } else {
          uint4* orow = reinterpret_cast<uint4*>(buf + r * 64);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(v[8 * u + 0], v[8 * u + 1]);
            w.y = pack_bf16x2(v[8 * u + 2], v[8 * u + 3]);
            w.z = pack_bf16x2(v[8 * u + 4], v[8 * u + 5]);
            w.w = pack_bf16x2(v[8 * u + 6], v[8 * u + 7]);
            orow[u] = w;
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (et == 0) {
          if (A2A)  // destination h's block, source q's rows (local), clipped at M/W and N/W
            tma_store_3d(&p.tmOut[ti.h], smem_u32(buf),
                         static_cast<int32_t>(ti.col0 - static_cast<int64_t>(ti.h) * p.g.Nw + cb * 32),
                         static_cast<int32_t>(ti.row0), ti.q);
          else
            tma_store_2d(&p.tmOut[0], smem_u32(buf), static_cast<int32_t>(ti.col0 + cb * 32),
                         static_cast<int32_t>(ti.row0));
          bulk_commit();
        }
        ++stage_ctr;
      }
      if (A2A && et == 0) {
        bulk_wait<0>();  // the tile's rows are in out_h before its chunks are counted
        fence_proxy_async_global();
      }
    }
#pragma unroll 1
    for (int cb = 0; cb < kBN / 32; ++cb) {
      if (tma_tile || c_tma) break;
      const int64_t c0 = ti.col0 + cb * 32;
      if (c0 >= ti.col_end) break;
      uint32_t v[32];
      tmem_ld32(tbase + cb * 32, v);
      if (!row_ok) continue;
      if (OP == kOpAG) {
        if (p.act) apply_activation(v, p.act);
        store_row32<kStoreF32>(p.out[0], p.ldc, row, c0, p.g.N, v);
      } else if (A2A) {
        if (fused_a2a)  // push: row q*Ms + row, column c0 - h*Nw of destination h's block
          store_row32<F32>(p.out[ti.h], p.ldc, static_cast<int64_t>(ti.q) * p.g.Ms + row,
                           c0 - static_cast<int64_t>(ti.h) * p.g.Nw, p.g.Nw, v);
        else            // baseline: into the rank's own Y_q
          store_row32<F32>(p.out[ti.q], p.ldc, row, c0, ti.col_end, v);
      } else if (!fused_rs) {  // baseline: partial of source q into slot [s][q]
        const size_t slot = static_cast<size_t>(s_row) * p.g.W + ti.q;
        store_row32<true>(p.recv + slot * static_cast<size_t>(p.g.Ms) * p.g.N, p.g.N, lr, c0,
                          p.g.N, v);
      } else if (in_order) {
        fold_row32<F32>(p, s_row, row, lr, d_row, c0, v);
      } else {  // park: an earlier partial of this unit is not folded yet
        store_row32<true>(park_ptr(p, s_row, d_row, 0, 0), p.g.N, lr, c0, p.g.N, v);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if constexpr (PAIR)
        mbar_arrive_cluster(acc ? tempty_bar1 : tempty_bar0);
      else
        mbar_arrive(L.tempty(acc));
    }
    ++tl;

    if (fused_a2a) {
      // notify: once all 128 rows are stored, count the tile on every chunk (h, q, j) its
      // rows touch; the last tile of a chunk releases the chunk's ready flag
      __threadfence();
      named_bar_sync(1, 128);
      if (et == 0 && ti.row_end > ti.row0) {
        const int32_t j0 = static_cast<int32_t>(ti.row0 / p.g.Cr);
        const int32_t j1 = static_cast<int32_t>((ti.row_end - 1) / p.g.Cr);
        for (int32_t j = j0; j <= j1; ++j) {
          const int64_t c = (static_cast<int64_t>(ti.h) * p.g.W + ti.q) * p.g.nC + j;
          const uint32_t old = atom_add_acq_rel_gpu(p.unit_cnt + c, 1u);
          if (old + 1u == static_cast<uint32_t>(a2a_chunk_tiles(p.g, j, kBM))) {
            p.unit_cnt[c] = 0u;  // ready for the next call
            st_release_gpu(p.ready + c, p.epoch);
          }
        }
      }
    }

    if (fused_rs) {
      // notify: publish this tile's fold or park of every piece
      __threadfence();
      named_bar_sync(1, 128);
      if (et == 0) {
        int k = 0;
        for (int64_t g = ti.row0; g < ti.row_end; ++k) {
          int32_t s, j;
          row_chunk(p.g, g, s, j);
          const int32_t d = fold_index(s, ti.q, p.g.W);
          uint32_t* word = words + k;
          int chain = -1;
          if ((L.last_mask[k >> 5] >> (k & 31)) & 1u) {
            if (d == p.g.W - 1) {
              *word = 0u;  // the unit is complete: ready for the next call
            } else {
              const uint32_t old = atom_add_acq_rel_gpu(word, 1u);
              if ((old >> (8 + d + 1)) & 1u) chain = d + 1;  // the next one is parked
            }
          } else {
            const uint32_t old = atom_or_acq_rel_gpu(word, 1u << (8 + d));
            if (static_cast<int32_t>(old & 0xffu) == d) chain = d;  // caught up meanwhile
          }
          L.chain[k] = static_cast<int8_t>(chain);
          g = static_cast<int64_t>(s) * p.g.Ms + min64(static_cast<int64_t>(j + 1) * p.g.Cr, p.g.Ms);
        }
      }
      named_bar_sync(1, 128);
      int k = 0;
      for (int64_t g = ti.row0; g < ti.row_end; ++k) {
        int32_t s, j;
        row_chunk(p.g, g, s, j);
        const int64_t hi = min64(ti.row_end, static_cast<int64_t>(s) * p.g.Ms +
                                                 min64(static_cast<int64_t>(j + 1) * p.g.Cr, p.g.Ms));
        const int chain = L.chain[k];
        if (chain >= 0) fold_chain<F32>(p, L, s, g, hi, ti.n, chain, words + k, et);
        g = hi;
      }
      named_bar_sync(1, 128);
    }
  }
  if (c_tma && et == 0) bulk_wait<0>();  // C's last boxes are in global memory
}

// ============================================================================ chunk transfer
// The piece's writes (bulk stores, complete; or the warp's fenced vector stores) are ordered
// before the count by the proxy fence and the count's release; the last piece's worker, which
// acquired every other count, releases the flag.
__device__ __forceinline__ void signal_piece(const KParams& p, int32_t c, int32_t total) {
  fence_proxy_async_global();
  const uint32_t old = atom_add_acq_rel_gpu(p.pieces_done + c, 1u);
  if (old + 1u == static_cast<uint32_t>(total)) {
    p.pieces_done[c] = 0u;
    st_release_gpu(p.ready + c, p.epoch);  // notify: chunk c has landed
    trace_min(p.trace, kTraceHead + 3 * static_cast<int64_t>(c));
  }
}

struct Piece {
  int32_t r0, nr;   // rows of the chunk
  int64_t boff;     // byte offset inside a row
  uint32_t nbytes;  // bytes per row copied
};

__device__ __forceinline__ Piece piece_of(const KParams& p, int32_t pc, int32_t rows_c) {
  Piece pc_;
  if (p.rows_per_piece > 0) {
    pc_.r0 = pc * p.rows_per_piece;
    pc_.nr = min32(p.rows_per_piece, rows_c - pc_.r0);
    pc_.boff = 0;
    pc_.nbytes = static_cast<uint32_t>(p.row_bytes);
  } else {
    pc_.r0 = pc / p.segs_per_row;
    pc_.nr = 1;
    const int32_t seg = pc - pc_.r0 * p.segs_per_row;
    pc_.boff = static_cast<int64_t>(seg) * p.piece_bytes;
    pc_.nbytes = static_cast<uint32_t>(min64(p.piece_bytes, p.row_bytes - pc_.boff));
  }
  return pc_;
}

// Pieces are numbered along the transfer order (chunk by chunk); worker w takes the pieces
// whose global number is w modulo the worker count, so every worker starts on the first
// chunk of the order.
template <typename Stop, typename F>
__device__ __forceinline__ void for_each_piece(const KParams& p, int32_t wid, int32_t nw,
                                               Stop&& stop, F&& f) {
  const int32_t nchunks = p.g.W * p.g.nC;
  const int64_t pieces_rank = static_cast<int64_t>(p.g.nC - 1) * p.pieces_full + p.pieces_last;
  for (int32_t tc = 0; tc < nchunks; ++tc) {
    if (stop()) return;
    int32_t s, j;
    ag_transfer_chunk(p.g, tc, s, j);
    const int32_t u = tc / p.g.nC;
    const int32_t rows_c =
        static_cast<int32_t>(min64(p.g.Cr, p.g.Ms - static_cast<int64_t>(j) * p.g.Cr));
    const int32_t total = (j == p.g.nC - 1) ? p.pieces_last : p.pieces_full;
    const int64_t base = static_cast<int64_t>(u) * pieces_rank +
                         static_cast<int64_t>(j) * p.pieces_full;
    const int32_t first = static_cast<int32_t>(((wid - base) % nw + nw) % nw);
    if (p.own_in_place && s == p.g.rank) continue;  // read in place, never transferred
    if (s * p.g.nC + j == p.drop_chunk) continue;     // the host dropped this message
    for (int32_t pc = first; pc < total; pc += nw) {
      if (!f(s, j, s * p.g.nC + j, total, piece_of(p, pc, rows_c))) return;
    }
  }
}

// One TMA bulk-copy worker (one thread): `nbuf` staging buffers of p.piece_bytes at `stage`,
// completion barriers bar0, bar0 + 8, ... (one per buffer).  Piece i goes through buffer
// i % nbuf; the worker keeps nbuf - 1 loads in flight and stores the oldest piece once its load
// has landed, so loads and stores overlap; a piece is counted towards its chunk once its
// store's writes are complete, which the worker checks kStoresInFlight stores later (it
// waits for a store's writes only when that many newer ones are outstanding).
struct CopyJob {
  uint8_t* dst;
  Piece pc;
  int32_t c, total;
};
constexpr uint32_t kMaxCopyBufs = 4;
constexpr uint32_t kDedicatedRingBytes = 12 * kCopyBuf;  // staging of a dedicated transfer CTA
constexpr int kStoresInFlight = 2;          // stores whose writes a worker does not wait for

static __device__ void run_copy_tma(const KParams& p, const SmemLayout& L, int32_t wid, int32_t nw,
                                    uint8_t* stage, uint32_t bar0, uint32_t nbuf) {
  uint32_t issued = 0;  // loads issued
  uint32_t stored = 0;  // loads waited for and their pieces' stores issued
  uint32_t counted = 0; // stored pieces counted towards their chunks
  CopyJob jobs[kMaxCopyBufs] = {};  // the piece in each buffer
  int32_t pend_c[kStoresInFlight + 1], pend_total[kStoresInFlight + 1];  // stored, not counted
  auto bar_of = [&](uint32_t i) { return bar0 + 8u * (i % nbuf); };
  auto buf_of = [&](uint32_t i) {
    return smem_u32(stage + (i % nbuf) * static_cast<uint32_t>(p.piece_bytes));
  };
  auto par_of = [&](uint32_t i) { return (i / nbuf) & 1u; };  // use i / nbuf of its barrier
  auto store_oldest = [&]() -> bool {
    const uint32_t i = stored;
    if (!wait_bar(p, L, bar_of(i), par_of(i), 500 + (i % nbuf))) return false;
    const CopyJob& job = jobs[i % nbuf];
    const uint32_t buf = buf_of(i);
    const uint32_t tot = job.pc.nbytes * static_cast<uint32_t>(job.pc.nr);
    if (job.pc.nbytes == static_cast<uint32_t>(p.row_bytes) || job.pc.nr == 1) {
      bulk_s2g(job.dst, buf, tot);  // gather rows are back to back (ld_gather == K)
    } else {
      for (int32_t r = 0; r < job.pc.nr; ++r)
        bulk_s2g(job.dst + static_cast<int64_t>(r) * p.ld_gather * 2, buf + r * job.pc.nbytes,
                 job.pc.nbytes);
    }
    bulk_commit();
    pend_c[stored % (kStoresInFlight + 1)] = job.c;
    pend_total[stored % (kStoresInFlight + 1)] = job.total;
    ++stored;
    if (stored - counted > static_cast<uint32_t>(kStoresInFlight)) {
      bulk_wait<kStoresInFlight>();  // the oldest uncounted piece's writes are complete
      signal_piece(p, pend_c[counted % (kStoresInFlight + 1)],
                   pend_total[counted % (kStoresInFlight + 1)]);
      ++counted;
    }
    return true;
  };
  auto stop = [&]() { return *L.abort_flag != 0; };
  for_each_piece(p, wid, nw, stop, [&](int32_t s, int32_t j, int32_t c, int32_t total,
                                       const Piece& pc) -> bool {
    const int64_t row_in_shard = static_cast<int64_t>(j) * p.g.Cr + pc.r0;
    const uint8_t* src = p.shard[s] + row_in_shard * p.lda_src * 2 + pc.boff;
    // buffer issued % nbuf was last read by the store of piece issued - nbuf, which has been
    // issued (at most nbuf - 1 pieces are loaded but not stored) and in steady state is the
    // newest store: wait until every issued store has read its shared memory
    bulk_wait_read<0>();
    const uint32_t i = issued;
    const uint32_t buf = buf_of(i), bar = bar_of(i);
    const uint32_t tot = pc.nbytes * static_cast<uint32_t>(pc.nr);
    mbar_expect_tx(bar, tot);
    if (p.src_rows_contig || pc.nr == 1) {
      bulk_g2s(buf, src, tot, bar);
    } else {
      for (int32_t r = 0; r < pc.nr; ++r)
        bulk_g2s(buf + r * pc.nbytes, src + static_cast<int64_t>(r) * p.lda_src * 2, pc.nbytes, bar);
    }
    jobs[i % nbuf] = {
        p.gather + (static_cast<int64_t>(s) * p.g.Ms + row_in_shard) * p.ld_gather * 2 + pc.boff,
        pc, c, total};
    ++issued;
    // keep nbuf - 1 loads in flight: store the oldest piece once nbuf are outstanding
    return issued - stored < nbuf || store_oldest();
  });
  while (!*L.abort_flag && stored < issued && store_oldest()) {
  }
  bulk_wait<0>();
  for (; !*L.abort_flag && counted < stored; ++counted)
    signal_piece(p, pend_c[counted % (kStoresInFlight + 1)],
                 pend_total[counted % (kStoresInFlight + 1)]);
  // after an abort, the loads still in flight (at most nbuf) land before the CTA can exit
  for (uint32_t i = stored; i < issued; ++i) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar_of(i), par_of(i)) && globaltimer_ns() - t0 < p.timeout_ns) {
    }
  }
}

// One vector ld/st copy worker (one warp).
constexpr int kLdstVecs = 16;
static __device__ void run_copy_ldst(const KParams& p, const SmemLayout& L, int lane, int32_t wid,
                                     int32_t nw) {
  // the whole warp takes the same decision
  auto stop = [&]() { return __shfl_sync(0xffffffffu, *L.abort_flag, 0) != 0; };
  for_each_piece(p, wid, nw, stop, [&](int32_t s, int32_t j, int32_t c, int32_t total,
                                       const Piece& pc) -> bool {
    const int64_t row_in_shard = static_cast<int64_t>(j) * p.g.Cr + pc.r0;
    const bool contig = pc.nr == 1 || (p.src_rows_contig && pc.nbytes == p.row_bytes);
    const int32_t nrow = contig ? 1 : pc.nr;
    const uint32_t nb = contig ? pc.nbytes * static_cast<uint32_t>(pc.nr) : pc.nbytes;
    for (int32_t r = 0; r < nrow; ++r) {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.shard[s] + (row_in_shard + r) * p.lda_src * 2 + pc.boff);
      uint4* dst = reinterpret_cast<uint4*>(
          p.gather + (static_cast<int64_t>(s) * p.g.Ms + row_in_shard + r) * p.ld_gather * 2 +
          pc.boff);
      // kLdstVecs vectors per lane in flight (8 KiB per warp): a copy at HBM rate needs tens
      // of KiB in flight per SM
      const int32_t nvec = static_cast<int32_t>(nb >> 4);
      for (int32_t v = lane; v < nvec; v += 32 * kLdstVecs) {
        uint4 x[kLdstVecs];
#pragma unroll
        for (int u = 0; u < kLdstVecs; ++u)
          if (v + u * 32 < nvec) x[u] = __ldg(src + v + u * 32);
#pragma unroll
        for (int u = 0; u < kLdstVecs; ++u)
          if (v + u * 32 < nvec) dst[v + u * 32] = x[u];
      }
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) signal_piece(p, c, total);
    __syncwarp();
    return true;
  });
}

// ============================================================================ kernel
// CL > 1: launched in clusters of CL CTAs that share each CL * 128-row tile (tcgen05
// cta_group::2 pairs); copy_ctas is then a multiple of CL, so dedicated transfer CTAs form
// whole clusters.
template <int OP, int COPY, bool F32, int CL>
__global__ void __launch_bounds__(kThreads, 1) fused_gemm_kernel(const __grid_constant__ KParams p) {
  static_assert(CL == 1 || CL == 2, "one CTA or a CTA pair per tile");
  constexpr bool PAIR = CL > 1;
  constexpr int NS = stages(PAIR);
  static_assert(COPY != kCopyTma ||
                    kDedicatedRingBytes <= NS * (kAStage + b_stage_bytes(PAIR)),
                "the dedicated TMA workers' buffers fit in the operand ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  SmemLayout L;
  L.ns = NS;
  L.a = base;
  L.b = L.a + NS * kAStage;
  L.copy = L.b + NS * b_stage_bytes(PAIR);
  uint8_t* misc = L.copy + 2 * kCopyBuf;
  L.bars = reinterpret_cast<uint64_t*>(misc);  // up to 32 barriers
  L.tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
  L.abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  L.unit_flag = reinterpret_cast<volatile int*>(misc + 264);
  L.vote = reinterpret_cast<volatile int*>(misc + 288);
  L.last_mask = reinterpret_cast<volatile uint32_t*>(misc + 320);
  L.chain = reinterpret_cast<volatile int8_t*>(misc + 384);
  L.ready_bits = reinterpret_cast<uint32_t*>(misc + 512);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < kReadyBitsWords) L.ready_bits[threadIdx.x] = 0u;
  const bool copier = static_cast<int32_t>(blockIdx.x) < p.copy_ctas;
  if (threadIdx.x == 0) {
    if (copier) {
      // a dedicated transfer CTA runs no GEMM: every barrier slot is a copy worker's
      for (int s = 0; s < 32; ++s) mbar_init(smem_u32(L.bars + s), 1);
    } else {
      for (int s = 0; s < NS; ++s) {
        mbar_init(L.full(s), 1);
        mbar_init(L.empty(s), 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(L.tfull(a), 1);
        mbar_init(L.tempty(a), PAIR ? 8 : 4);  // the epilogue warps of the tile's CTA(s)
        mbar_init(L.copyb(a), 1);
      }
      mbar_init(L.fin(), 1);
    }
    *L.abort_flag = 0;
    *L.unit_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA[0]);
    tma_prefetch_desc(&p.tmB[0]);
  }
  if (warp == 1 && !copier) {
    if constexpr (PAIR) tmem_alloc_pair(smem_u32(L.tmem_slot), kTmemCols);
    else tmem_alloc(smem_u32(L.tmem_slot), kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the cluster's barriers exist before any CTA signals them
  tc_fence_after();
  const uint32_t tmem_base = copier ? 0u : *L.tmem_slot;
  // everything above touches only shared memory, TMEM and the parameter space, so it may
  // overlap the grid before this one (launched with programmatic stream serialization after
  // the prepare kernel); no global memory is read or written before that grid has completed
  griddep_wait();
  if (threadIdx.x == 0) trace_min(p.trace, 0);

  if (copier) {
    // dedicated transfer CTA: no GEMM; the operand ring becomes four workers' staging rings
    // of ded_bufs piece-sized buffers each: as many workers (one per warp, at most 8) as the
    // 192 KiB of the ring hold
    if (OP == kOpAG && !p.plain) {
      const uint32_t nbuf = static_cast<uint32_t>(p.ded_bufs);
      const int nwk = min32(8, static_cast<int32_t>(kDedicatedRingBytes /
                                                    (static_cast<uint32_t>(p.piece_bytes) * nbuf)));
      if (COPY == kCopyTma && warp < nwk && lane == 0)
        run_copy_tma(p, L, static_cast<int32_t>(blockIdx.x) * nwk + warp, p.copy_ctas * nwk,
                     L.a + warp * nbuf * p.piece_bytes, smem_u32(L.bars + warp * nbuf), nbuf);
      if (COPY == kCopyLdst)
        run_copy_ldst(p, L, lane, static_cast<int32_t>(blockIdx.x) * 8 + warp, p.copy_ctas * 8);
    }
  } else if (warp == 0) {
    run_producer<OP, CL, NS>(p, L);
  } else if (warp == 1) {
    if ((cl_rank<CL>() & 1u) == 0u) run_mma<OP, CL, NS>(p, L, tmem_base);
  } else if (warp < 4) {
    if (OP == kOpAG && !p.plain && p.copy_ctas == 0) {  // co-located transfer warps
      if (COPY == kCopyTma && warp == 2 && lane == 0)
        run_copy_tma(p, L, static_cast<int32_t>(blockIdx.x), static_cast<int32_t>(gridDim.x),
                     L.copy, L.copyb(0), 2);
      if (COPY == kCopyLdst)
        run_copy_ldst(p, L, lane, static_cast<int32_t>(blockIdx.x) * 2 + (warp - 2),
                      static_cast<int32_t>(gridDim.x) * 2);
    }
  } else {
    run_epilogue<OP, F32, CL>(p, L, tmem_base, warp, lane, COPY != kCopyTma || p.copy_ctas > 0);
  }

  tc_fence_before();
  __syncthreads();
  // no CTA of a cluster leaves while another may still read or write its shared memory or TMEM
  if constexpr (PAIR) cluster_sync();
  if (warp == 1 && !copier) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
  // the next call's prepare kernel (stream-ordered after this grid) may then skip rewriting
  // the tile order and clearing the control arrays
  if (p.tag != nullptr && blockIdx.x == 0 && threadIdx.x == 0 && *(volatile uint32_t*)p.err == 0u)
    *p.tag = p.tag_value;
  if (p.trace != nullptr && threadIdx.x == 0)
    atomicMax(p.trace + 1, static_cast<unsigned long long>(globaltimer_ns()));
}

}  // namespace dt
