// C ABI of the fused AllGather-GEMM / GEMM-ReduceScatter (declared in include/dt.h).
//
// Host responsibilities: argument validation, workspace layout, the per-workspace call
// epoch (so ready flags never need resetting), tensor-map encoding, the plan kernel, the
// copy-engine chunk transfer, kernel launches, and the kernel-level-overlap baselines.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "dt.h"
#include "dt_internal.h"

using namespace dt;

namespace {

// ------------------------------------------------------------------------------ errors
thread_local std::string g_last_error;

dt_status fail(dt_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

dt_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define DT_CUDA(call)                                    \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);  \
  } while (0)

// One NVTX range per library call (named after the call), visible to a profiler's timeline;
// without a tool attached the push and pop do nothing.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ------------------------------------------------------------------------------ driver entry points
typedef CUresult (*PfnEncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*PfnWriteValue32)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

void* driver_fn(const char* name) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return fn;
}

PfnEncodeTiled encode_tiled() {
  static PfnEncodeTiled fn = reinterpret_cast<PfnEncodeTiled>(driver_fn("cuTensorMapEncodeTiled"));
  return fn;
}
PfnWriteValue32 write_value32() {
  static PfnWriteValue32 fn = reinterpret_cast<PfnWriteValue32>(driver_fn("cuStreamWriteValue32"));
  return fn;
}

// 2-D bf16 tensor map with 128-byte swizzle: `inner` contiguous elements per row, `outer`
// rows `row_stride_bytes` apart; boxes of box_inner x box_outer elements.
dt_status make_tmap(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  PfnEncodeTiled enc = encode_tiled();
  if (!enc) return fail(DT_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(tm, dtype, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %llu x %llu, stride %llu",
                static_cast<int>(r), (unsigned long long)inner, (unsigned long long)outer,
                (unsigned long long)row_stride_bytes);
  return DT_OK;
}

// ------------------------------------------------------------------------------ derived problem
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Derived {
  int op;
  int32_t W, rank, G, Tm, Tn, KB, T, nC, pieces_max;
  int32_t bm;    // rows of a tile in the order: 128 (one CTA), 256 (a CTA pair)
  int32_t cl;    // CTAs per cluster: bm / 128
  int32_t Tm128; // 128-row m-tiles (one CTA's rows): the ReduceScatter's unit granularity
  int64_t M, N, K, Ms, Cr, lda, ldb, ldc, ld_gather;
  bool swizzle, f32;
  int backend;  // resolved for AG
  int32_t copy_ctas;
  int32_t act;
  uint64_t timeout_ns;
  Geom geom;
  size_t off_ready, off_pieces, off_cnt, off_order, ctl_bytes, off_data, total;
};

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

uint64_t default_timeout_ns() {
  static uint64_t v = [] {
    const char* e = getenv("DT_WAIT_TIMEOUT_US");
    long long us = e ? atoll(e) : 0;
    if (us <= 0) us = 2000000;
    return static_cast<uint64_t>(us) * 1000ull;
  }();
  return v;
}

// TMA buffers per worker on a dedicated transfer CTA (1 to 4); DT_COPY_BUFS overrides.
// Measured on 256 MiB AllGathers at 2048-row chunks (L2 flushed): 32 KiB pieces, 6 workers x 1
// buffer 5.79-5.91 TB/s, 3 x 2 5.54-5.66; 16 KiB pieces, 8 x 1 5.54, 6 x 2 5.48-5.54, 4 x 3
// 5.16-5.26, 3 x 4 4.87; 8 KiB pieces 4.35-4.65; a ring per warp pair with separate loader and
// storer threads 4.67-4.96.  More workers and bigger pieces win: a worker's serial per-piece
// work, not the bytes in flight, sets the rate.
int32_t ded_bufs_setting() {
  static int32_t v = [] {
    const char* e = getenv("DT_COPY_BUFS");
    const int x = e ? atoi(e) : 1;
    return static_cast<int32_t>(x < 1 ? 1 : (x > 4 ? 4 : x));
  }();
  return v;
}

// Bytes of a transfer piece on dedicated transfer CTAs (8, 16 or 32 KiB); DT_COPY_PIECE
// overrides (see the measurements above).
int32_t ded_piece_setting() {
  static int32_t v = [] {
    const char* e = getenv("DT_COPY_PIECE");
    const int x = e ? atoi(e) : 32768;
    return static_cast<int32_t>(x <= 8192 ? 8192 : (x >= 32768 ? 2 * kCopyBuf : kCopyBuf));
  }();
  return v;
}

// The fused AllGather-GEMM stores C through TMA (1) or per thread (0); DT_C_TMA overrides.
int32_t c_tma_setting() {
  static int32_t v = [] {
    const char* e = getenv("DT_C_TMA");
    return e ? (atoi(e) != 0 ? 1 : 0) : 1;
  }();
  return v;
}

// C's tensor map for the TMA-store epilogue: 32-column x 128-row boxes; bf16 boxes are dense
// 64-byte rows, fp32 boxes 128-byte rows in the 128-byte swizzle.
dt_status make_c_tmap(CUtensorMap* tm, void* c, int64_t rows, int64_t cols, int64_t ldc, bool f32);

// Bytes of B_q that one column band of the ReduceScatter order may use (automatic col_band).
constexpr int64_t kBandBytes = 32ll << 20;

// ReduceScatter / AllReduce middle sources fold with a TMA reduce-add (1) or a load, add and
// store (0); DT_RS_REDUCE overrides.
int32_t rs_reduce_setting() {
  static int32_t v = [] {
    const char* e = getenv("DT_RS_REDUCE");
    return e ? (atoi(e) != 0 ? 1 : 0) : 1;
  }();
  return v;
}

// Per-wave rotation of the CTAs' slots in the tile order (KParams::rot) of the ReduceScatter and
// AllReduce, whose tiles cut by destination boundaries fold at a higher cost and recur at fixed
// slots of a wave: one slot per wave; DT_ROT overrides (0: every CTA takes the same slot of
// every wave, as the AllGather and AllToAll do, whose tiles cost alike).
int32_t rot_setting() {
  static int32_t v = [] {
    const char* e = getenv("DT_ROT");
    const int x = e ? atoi(e) : 1;
    return static_cast<int32_t>(x < 0 ? 0 : x);
  }();
  return v;
}

// L2 cache policies of the fused kernels (KParams::l2_hints); DT_L2_HINTS overrides.
int32_t l2_hints_setting() {
  static int32_t v = [] {
    const char* e = getenv("DT_L2_HINTS");
    return e ? static_cast<int32_t>(atoi(e)) & 3 : 3;
  }();
  return v;
}

dt_status derive(const dt_args* a, int op, Derived* d) {
  if (!a) return fail(DT_ERR_INVALID, "args is NULL");
  if (op != DT_OP_AG_GEMM && op != DT_OP_GEMM_RS && op != DT_OP_GEMM_AR && op != DT_OP_GEMM_A2A)
    return fail(DT_ERR_INVALID, "unknown op %d", op);
  const bool a2a = op == DT_OP_GEMM_A2A;
  d->op = op;
  d->W = a->world_size;
  if (d->W < 1 || d->W > DT_MAX_WORLD)
    return fail(DT_ERR_INVALID, "world_size %d outside 1..%d", d->W, DT_MAX_WORLD);
  d->rank = a->rank;
  if (op == DT_OP_AG_GEMM && (d->rank < 0 || d->rank >= d->W))
    return fail(DT_ERR_INVALID, "rank %d outside 0..%d", d->rank, d->W - 1);
  if (op != DT_OP_AG_GEMM) d->rank = 0;
  d->M = a->m;
  d->N = a->n;
  d->K = a->k;
  if (d->M < 0 || d->N < 0 || d->K < 0) return fail(DT_ERR_INVALID, "negative size");
  if (d->M >= (1ll << 31) || d->N >= (1ll << 31) || d->K >= (1ll << 31))
    return fail(DT_ERR_UNSUPPORTED, "sizes must be below 2^31");
  if (d->M % d->W) return fail(DT_ERR_INVALID, "M=%lld is not a multiple of W=%d", (long long)d->M, d->W);
  if (d->N % 8) return fail(DT_ERR_UNSUPPORTED, "N=%lld must be a multiple of 8", (long long)d->N);
  if (op == DT_OP_AG_GEMM && d->K % 8)
    return fail(DT_ERR_UNSUPPORTED, "AllGather K=%lld must be a multiple of 8", (long long)d->K);
  if (a2a && d->N % d->W)
    return fail(DT_ERR_INVALID, "AllToAll N=%lld is not a multiple of W=%d", (long long)d->N, d->W);
  if (a2a && (d->N / d->W) % 8)
    return fail(DT_ERR_UNSUPPORTED, "AllToAll N/W=%lld must be a multiple of 8 (16-byte column blocks)",
                (long long)(d->N / d->W));
  d->Cr = a->chunk_rows;
  if (d->Cr < 1) return fail(DT_ERR_INVALID, "chunk_rows must be >= 1");
  d->lda = a->lda ? a->lda : d->K;
  d->ldb = a->ldb ? a->ldb : d->N;
  const int64_t out_cols = a2a ? d->N / d->W : d->N;  // columns of each output
  d->ldc = a->ldc ? a->ldc : out_cols;
  if (d->lda < d->K || d->ldb < d->N || d->ldc < out_cols)
    return fail(DT_ERR_INVALID, "leading dimension smaller than the row length");
  if ((d->lda % 8) || (d->ldb % 8) || (d->ldc % 8))
    return fail(DT_ERR_INVALID, "leading dimensions must be multiples of 8 elements (16-byte rows)");
  if ((a->tile_m != 0 && a->tile_m != kBM && a->tile_m != 2 * kBM) ||
      (a->tile_n != 0 && a->tile_n != kBN))
    return fail(DT_ERR_UNSUPPORTED, "tiles other than %d or %d x %d are not built", kBM, 2 * kBM,
                kBN);
  if (a->out_dtype != DT_BF16 && a->out_dtype != DT_F32)
    return fail(DT_ERR_INVALID, "unknown out_dtype %d", a->out_dtype);
  d->f32 = a->out_dtype == DT_F32;
  d->swizzle = a->swizzle != 0;
  d->G = a->group > 0 ? a->group : 8;
  d->timeout_ns = a->timeout_us > 0 ? static_cast<uint64_t>(a->timeout_us) * 1000ull
                                    : default_timeout_ns();
  d->Ms = d->M / d->W;
  // tile rows: as asked, or a CTA pair (256 rows) when that still gives every pair of SMs a
  // tile (at least 76 pair tiles), else one CTA (128 rows)
  const int64_t rows_tiled = a2a ? d->Ms : d->M;  // rows one rank's tiles cover
  const int64_t copies = op == DT_OP_AG_GEMM ? 1 : d->W;
  if (a->tile_m != 0) {
    d->bm = a->tile_m;
  } else {
    const int64_t t256 = copies * cdiv64(rows_tiled, 2 * kBM) * cdiv64(a2a ? d->N / d->W : d->N, kBN) *
                         (a2a ? d->W : 1);
    const bool odd_copiers = op == DT_OP_AG_GEMM && (a->copy_ctas % 2) != 0;
    d->bm = t256 >= 76 && !odd_copiers ? 2 * kBM : kBM;
  }
  d->cl = d->bm / kBM;
  d->Tm128 = static_cast<int32_t>(cdiv64(rows_tiled, kBM));
  d->geom = a2a ? make_geom_a2a(d->W, d->M, d->N, d->Cr, d->bm, kBN, d->G, d->swizzle ? 1 : 0)
              : make_geom(d->W, d->rank, d->M, d->N, d->Cr, d->bm, kBN, d->G, d->swizzle ? 1 : 0);
  if (a->col_band < 0) return fail(DT_ERR_INVALID, "col_band must be >= 0");
  if (op != DT_OP_GEMM_A2A) {
    // column bands: one band of B (K x band columns, bf16) within kBandBytes, so that it stays
    // in L2 while the order visits every destination (ReduceScatter) or chunk (AllGather)
    const int32_t tn = d->geom.Tn;
    int32_t nb = a->col_band;
    if (nb == 0) {
      const int64_t b_bytes = d->K * d->N * 2;
      const int64_t bands = std::max<int64_t>(1, cdiv64(b_bytes, kBandBytes));
      nb = static_cast<int32_t>(cdiv64(tn, std::min<int64_t>(bands, std::max(tn, 1))));
    }
    d->geom.Nb = std::max(1, std::min(nb, std::max(tn, 1)));
  }
  d->nC = d->geom.nC;
  d->Tm = d->geom.Tm;
  d->Tn = d->geom.Tn;
  d->KB = static_cast<int32_t>(cdiv64(d->K, kBK));
  const int64_t T64 = (op == DT_OP_AG_GEMM ? 1 : d->W) * static_cast<int64_t>(d->Tm) * d->Tn;
  if (T64 >= (1ll << 31)) return fail(DT_ERR_UNSUPPORTED, "too many tiles");
  d->T = static_cast<int32_t>(T64);
  if ((op == DT_OP_GEMM_RS || op == DT_OP_GEMM_AR) && static_cast<int64_t>(d->W - 1) * d->M >= (1ll << 31))
    return fail(DT_ERR_UNSUPPORTED, "(W-1)*M must be below 2^31");
  if (static_cast<int64_t>(d->W) * d->W * d->nC >= (1ll << 24))
    return fail(DT_ERR_UNSUPPORTED, "too many chunks; raise chunk_rows");
  d->ld_gather = d->K;  // K % 8 == 0: 16-byte rows, back to back
  int be = a->backend;
  if (be < DT_XFER_AUTO || be > DT_XFER_TMA_TILE)
    return fail(DT_ERR_INVALID, "unknown backend %d", be);
  if (be == DT_XFER_TMA_TILE) {
    if (op != DT_OP_AG_GEMM)
      return fail(DT_ERR_INVALID, "DT_XFER_TMA_TILE applies to the AllGather-GEMM only");
    if (d->Ms % kBM)
      return fail(DT_ERR_UNSUPPORTED,
                  "DT_XFER_TMA_TILE needs M/W (%lld) to be a multiple of %d (no tile across shards)",
                  (long long)d->Ms, kBM);
    if (a->copy_ctas != 0) return fail(DT_ERR_INVALID, "DT_XFER_TMA_TILE uses no transfer CTAs");
  }
  if (op == DT_OP_AG_GEMM && be == DT_XFER_AUTO) {
    // large chunks amortise the copy engine's per-transfer launch cost; smaller ones move
    // on in-kernel TMA bulk copies
    const int64_t chunk_bytes = std::min<int64_t>(d->Cr, d->Ms) * d->K * 2;
    be = chunk_bytes >= (8ll << 20) && a->copy_ctas == 0 ? DT_XFER_COPY_ENGINE : DT_XFER_TMA;
  }
  d->backend = be;
  if (a->act < DT_ACT_NONE || a->act > DT_ACT_SILU) return fail(DT_ERR_INVALID, "unknown act %d", a->act);
  if (a->act != DT_ACT_NONE && op != DT_OP_AG_GEMM)
    return fail(DT_ERR_UNSUPPORTED, "activations apply to the AllGather-GEMM only");
  d->act = a->act;
  d->copy_ctas = op == DT_OP_AG_GEMM ? a->copy_ctas : 0;
  if (d->copy_ctas < 0 || d->copy_ctas > 64)
    return fail(DT_ERR_INVALID, "copy_ctas %d outside 0..64", d->copy_ctas);
  if (d->copy_ctas > 0 && be == DT_XFER_COPY_ENGINE)
    return fail(DT_ERR_INVALID, "dedicated transfer CTAs need DT_XFER_TMA or DT_XFER_LDST");
  if (d->copy_ctas % d->cl)
    return fail(DT_ERR_INVALID, "copy_ctas must be a multiple of the %d CTAs of a %d-row tile",
                d->cl, d->bm);
  // workspace layout: error word | control arrays | tile order || data
  const size_t nchunks = static_cast<size_t>(d->W) * d->nC;
  size_t off = 256;
  d->off_ready = d->off_pieces = d->off_cnt = 0;
  d->pieces_max = 0;
  if (op == DT_OP_AG_GEMM) {
    d->off_ready = off;
    off = align_up(off + 4 * nchunks, 256);
    d->off_pieces = off;
    off = align_up(off + 4 * nchunks, 256);
  } else if (a2a) {
    // per (destination h, source q, chunk j): count of stored tiles, then the ready flag
    d->off_cnt = off;
    off = align_up(off + 4 * nchunks * d->W, 256);
    d->off_ready = off;
    off = align_up(off + 4 * nchunks * d->W, 256);
  } else {
    // reduction units live on one CTA's 128 rows, whatever the tile of the order
    const Geom g128 = make_geom(d->W, 0, d->M, d->N, d->Cr, kBM, kBN, d->G, 1);
    d->pieces_max = d->Tm128 > 0 && d->Ms > 0 ? rs_pieces_max(g128) : 0;
    d->off_cnt = off;
    off = align_up(off + 4 * static_cast<size_t>(d->Tm128) * d->Tn * d->pieces_max, 256);
  }
  d->off_order = off;
  off = align_up(off + 4 * static_cast<size_t>(d->T), 1024);
  d->ctl_bytes = off;
  d->off_data = off;
  if (op == DT_OP_AG_GEMM && be != DT_XFER_TMA_TILE)
    d->total = off + static_cast<size_t>(d->M) * d->ld_gather * 2;
  else if (op == DT_OP_AG_GEMM)
    d->total = off;  // the tiles read the shards in place: no gather buffer
  else if (a2a)
    d->total = off;
  else
    d->total = off + static_cast<size_t>(d->W) * d->W * d->Ms * d->N * 4;
  return DT_OK;
}

// ------------------------------------------------------------------------------ per-workspace state
struct LayoutKey {
  int op, W, rank, G, swz, bm, nb;
  long long M, N, K, Cr;
};

struct WsState {
  uint32_t epoch;
};

std::mutex g_mu;
std::map<const void*, WsState> g_ws;

// host-side fault injection for failure-detection tests: transfer step whose copy and flag
// write the next AllGather call leaves out (-1: none)
int32_t g_drop_transfer = -1;

// debug timeline of the fused AllGather-GEMM calls (dt_trace_attach), caller-owned device
// memory; null when tracing is off
std::mutex g_trace_mu;
void* g_trace = nullptr;
size_t g_trace_bytes = 0;

size_t trace_bytes_for(int32_t W, int32_t nC) {
  return (static_cast<size_t>(kTraceHead) + 3 * static_cast<size_t>(W) * nC) * 8;
}

LayoutKey key_of(const Derived& d) {
  return LayoutKey{d.op, d.W, d.rank, d.G, d.swizzle ? 1 : 0, d.bm, d.geom.Nb, d.M, d.N, d.K, d.Cr};
}

// 64-bit tag of the workspace layout (FNV-1a over the key), never 0
unsigned long long layout_tag(const Derived& d) {
  const LayoutKey k = key_of(d);
  const long long v[11] = {k.op, k.W, k.rank, k.G, k.swz, k.bm, k.nb, k.M, k.N, k.K, k.Cr};
  unsigned long long h = 1469598103934665603ull;
  for (long long x : v) {
    for (int b = 0; b < 8; ++b) {
      h ^= static_cast<unsigned long long>((x >> (8 * b)) & 0xff);
      h *= 1099511628211ull;
    }
  }
  return h | 1ull;
}

constexpr size_t kTagOffset = 16;  // after the 4-word error block

// Bring the workspace to this call: bump the host-side epoch and launch the prepare kernel,
// which rewrites the tile order and clears the control arrays unless the workspace already
// carries this layout's tag and no recorded error.
dt_status prepare_workspace(const Derived& d, void* ws, cudaStream_t stream, uint32_t* epoch);

// ------------------------------------------------------------------------------ device info
// Copy-engine chunk copies are spread round-robin over this many streams: one stream moves
// 8 MiB device-to-device copies at ~2.7 TB/s (read + write), four at ~5 TB/s.
constexpr int kCopyStreams = 4;

struct DevCtx {
  int sms = 0;
  cudaStream_t side = nullptr;
  cudaStream_t copy[kCopyStreams] = {};
  cudaEvent_t copy_done[kCopyStreams] = {};
  cudaEvent_t ev_start = nullptr, ev_done = nullptr;
  cudaEvent_t tune_t0 = nullptr, tune_t1 = nullptr;  // timing events of the tuner
  std::vector<cudaEvent_t> chunk_events;
};
std::mutex g_dev_mu;
std::map<int, DevCtx> g_dev;

dt_status dev_ctx(DevCtx** out) {
  int dev = 0;
  DT_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevCtx& c = g_dev[dev];
  if (c.sms == 0) {
    // sms is set last: a set-up that fails part way is redone by the next call
    int sms = 0;
    DT_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (!c.side) DT_CUDA(cudaStreamCreateWithFlags(&c.side, cudaStreamNonBlocking));
    for (int i = 0; i < kCopyStreams; ++i) {
      if (!c.copy[i]) DT_CUDA(cudaStreamCreateWithFlags(&c.copy[i], cudaStreamNonBlocking));
      if (!c.copy_done[i]) DT_CUDA(cudaEventCreateWithFlags(&c.copy_done[i], cudaEventDisableTiming));
    }
    if (!c.ev_start) DT_CUDA(cudaEventCreateWithFlags(&c.ev_start, cudaEventDisableTiming));
    if (!c.ev_done) DT_CUDA(cudaEventCreateWithFlags(&c.ev_done, cudaEventDisableTiming));
    c.sms = sms;
  }
  *out = &c;
  return DT_OK;
}

// The copy streams start after `stream`'s work so far (fork) and `stream` continues after
// theirs (join); the caller holds g_dev_mu in between.
dt_status fork_copies(DevCtx* dev, cudaStream_t stream) {
  DT_CUDA(cudaEventRecord(dev->ev_start, stream));
  for (int i = 0; i < kCopyStreams; ++i) DT_CUDA(cudaStreamWaitEvent(dev->copy[i], dev->ev_start, 0));
  return DT_OK;
}
dt_status join_copies(DevCtx* dev, cudaStream_t stream) {
  for (int i = 0; i < kCopyStreams; ++i) {
    DT_CUDA(cudaEventRecord(dev->copy_done[i], dev->copy[i]));
    DT_CUDA(cudaStreamWaitEvent(stream, dev->copy_done[i], 0));
  }
  return DT_OK;
}

// ------------------------------------------------------------------------------ small kernels
__global__ void plan_kernel(Geom g, int op, int32_t* order, int32_t T) {
  const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int64_t pos = tile_position(g, op, t);
  if (pos >= 0 && pos < T) order[pos] = t;
}

// Once per call before the fused kernel: if the workspace does not carry `tag` (new or
// zero-filled memory, another problem, or a call that recorded an error), write the tile
// order and zero the per-chunk flags and counters.  All blocks read the tag before anyone
// can change it: only the fused kernel writes it, after this grid has finished.
__global__ void prepare_kernel(Geom g, int op, int32_t* order, int32_t T, uint32_t* ctl,
                               int64_t ctl_words, const uint32_t* err,
                               const unsigned long long* tag, unsigned long long expected) {
  // the fused kernel behind this grid may start launching now: it waits for this grid's
  // completion before it reads or writes global memory
  griddep_launch_dependents();
  if (*tag == expected && err[0] == 0u) return;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  for (int64_t w = t0; w < ctl_words; w += stride) ctl[w] = 0u;
  for (int64_t t = t0; t < T; t += stride) {
    const int64_t pos = tile_position(g, op, t);
    if (pos >= 0 && pos < T) order[pos] = static_cast<int32_t>(t);
  }
}

__global__ void zero_rows_kernel(uint8_t* dst, int64_t rows, int64_t row_bytes, int64_t ld_bytes) {
  const int64_t nv = row_bytes / 16;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < rows * nv;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e / nv, v = e - r * nv;
    reinterpret_cast<uint4*>(dst + r * ld_bytes)[v] = make_uint4(0, 0, 0, 0);
  }
}

// out_s = the fp32 partial slots recv[s][q] summed in the fused path's fixed source order
// q = 0..W-1
struct OutRows {
  void* p[DT_MAX_WORLD];  // ReduceScatter: out_s; AllReduce: every rank's output
  int32_t n;
  int64_t row0;            // first output row of this destination block
};

__global__ void reduce_slots_kernel(const float* recv, int32_t W, int64_t Ms, int64_t N, int32_t s,
                                    OutRows out, int64_t ldc, int f32) {
  const int64_t nv = N / 4;
  const size_t slot = static_cast<size_t>(Ms) * N;
  const float* base = recv + static_cast<size_t>(s) * W * slot;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < Ms * nv;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e / nv, v = e - r * nv;
    const float* src = base + r * N + v * 4;
    float4 acc = __ldcg(reinterpret_cast<const float4*>(src));
    for (int32_t q = 1; q < W; ++q) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(src + q * slot));
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&lo);
    w.y = *reinterpret_cast<uint32_t*>(&hi);
    for (int32_t c = 0; c < out.n; ++c) {
      const int64_t row = out.row0 + r;
      if (f32)
        reinterpret_cast<float4*>(reinterpret_cast<float*>(out.p[c]) + row * ldc)[v] = acc;
      else
        reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out.p[c]) + row * ldc)[v] = w;
    }
  }
}

dt_status launch_zero(void* dst, int64_t rows, int64_t row_bytes, int64_t ld_bytes,
                      cudaStream_t stream) {
  if (rows <= 0 || row_bytes <= 0) return DT_OK;
  const int64_t work = rows * (row_bytes / 16);
  const int grid = static_cast<int>(std::min<int64_t>(cdiv64(work, 256), 4096));
  zero_rows_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<uint8_t*>(dst), rows, row_bytes,
                                             ld_bytes);
  DT_CUDA(cudaGetLastError());
  return DT_OK;
}

// The prepare kernel of one call on `ws` (see prepare_kernel).
dt_status launch_prepare(const Derived& d, void* ws, cudaStream_t stream) {
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  const size_t ctl_begin = 256;
  const int64_t ctl_words = static_cast<int64_t>((d.off_order - ctl_begin) / 4);
  const int64_t work = std::max<int64_t>(d.T, ctl_words);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(std::max<int64_t>(cdiv64(work, 256), 1), 1024));
  prepare_kernel<<<grid, 256, 0, stream>>>(
      d.geom, d.op, reinterpret_cast<int32_t*>(w + d.off_order), d.T,
      reinterpret_cast<uint32_t*>(w + ctl_begin), ctl_words, reinterpret_cast<uint32_t*>(w),
      reinterpret_cast<unsigned long long*>(w + kTagOffset), layout_tag(d));
  DT_CUDA(cudaGetLastError());
  return DT_OK;
}

dt_status prepare_workspace(const Derived& d, void* ws, cudaStream_t stream, uint32_t* epoch) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    WsState& st = g_ws[ws];
    if (++st.epoch == 0u) st.epoch = 1u;  // ready flags hold epochs; 0 means "never"
    *epoch = st.epoch;
  }
  return launch_prepare(d, ws, stream);
}

// The transfer step that dt_debug_drop_transfer asked the next AllGather to leave out (-1:
// none); reading it clears it.
int32_t take_drop_transfer() {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  const int32_t drop = g_drop_transfer;
  g_drop_transfer = -1;
  return drop;
}

// The in-kernel transfer leaves out the chunk of transfer step `drop` (no copy, no flag).
void set_drop_chunk(KParams& p, const Derived& d, int32_t drop) {
  if (drop < 0 || drop >= d.W * d.nC) return;
  int32_t s, j;
  ag_transfer_chunk(d.geom, drop, s, j);
  p.drop_chunk = s * d.nC + j;
}

// out_h of the AllToAll as a 3-D tensor [W sources][M/W rows][N/W columns]: a box stored at
// (x, y, source q) is clipped at source q's rows and at the destination's columns.
dt_status make_a2a_out_tmap(CUtensorMap* tm, void* out, int64_t ms, int64_t nw, int64_t ldc,
                            int32_t w, bool f32) {
  PfnEncodeTiled enc = encode_tiled();
  if (!enc) return fail(DT_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const uint64_t esz = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(nw), static_cast<cuuint64_t>(ms),
                              static_cast<cuuint64_t>(w)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldc) * esz,
                                 static_cast<cuuint64_t>(ms) * ldc * esz};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(kBM), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(DT_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for the AllToAll output", (int)r);
  return DT_OK;
}

dt_status make_c_tmap(CUtensorMap* tm, void* c, int64_t rows, int64_t cols, int64_t ldc, bool f32) {
  return make_tmap(tm, c, cols, rows, static_cast<uint64_t>(ldc) * (f32 ? 4 : 2), 32, kBM,
                   f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

dt_status check_ws(const Derived& d, void* ws, size_t bytes) {
  if (!ws) return fail(DT_ERR_WORKSPACE, "workspace is NULL");
  if (!is_aligned(ws, 256)) return fail(DT_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (bytes < d.total)
    return fail(DT_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", bytes, d.total);
  return DT_OK;
}

// Persistent grid over `tiles` tiles of the order with `sms` SMs to use: one CTA per SM, or
// one cluster of two per pair of SMs.
int grid_for(const Derived& d, int64_t tiles, int sms) {
  return d.cl * static_cast<int>(std::min<int64_t>(tiles, std::max(sms / d.cl, 1)));
}

void fill_common(KParams& p, const Derived& d, void* ws, uint32_t epoch) {
  memset(&p, 0, sizeof(p));
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  p.err = reinterpret_cast<uint32_t*>(w);
  p.tag = reinterpret_cast<unsigned long long*>(w + kTagOffset);
  p.tag_value = layout_tag(d);
  p.order = reinterpret_cast<const int32_t*>(w + d.off_order);
  p.g = d.geom;
  p.ldc = d.ldc;
  p.row_lo = 0;
  p.row_hi = d.M;
  p.Tm = d.Tm;
  p.KB = d.KB;
  p.T = d.T;
  p.epoch = epoch;
  p.timeout_ns = d.timeout_ns;
  p.act = d.act;
  p.drop_chunk = -1;
  p.l2_hints = l2_hints_setting();
  p.rs_reduce = rs_reduce_setting();
  p.trace = nullptr;
  p.ded_bufs = ded_bufs_setting();
  p.piece_bytes = kCopyBuf;
}

// Point the kernel at the attached timeline (if any) and reset it on `stream`: the min words to
// all ones, the sums to zero.
dt_status attach_trace(KParams& p, const Derived& d, cudaStream_t stream) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (g_trace == nullptr) return DT_OK;
  const size_t need = trace_bytes_for(d.W, d.nC);
  if (g_trace_bytes < need)
    return fail(DT_ERR_INVALID, "the attached trace buffer holds %zu bytes, this call needs %zu",
                g_trace_bytes, need);
  DT_CUDA(cudaMemsetAsync(g_trace, 0xff, need, stream));
  DT_CUDA(cudaMemsetAsync(reinterpret_cast<uint8_t*>(g_trace) + 8, 0, 24, stream));
  p.trace = reinterpret_cast<unsigned long long*>(g_trace);
  return DT_OK;
}

// ------------------------------------------------------------------------------ AllGather
// How the in-kernel transfer cuts a chunk into pieces of at most one 16 KiB staging buffer:
// whole rows when a row fits (rows_per_piece of them), else 16 KiB segments of one row.
void set_pieces(KParams& p, const Derived& d, bool dedicated) {
  p.row_bytes = d.K * 2;
  p.piece_bytes = dedicated ? ded_piece_setting() : kCopyBuf;
  if (p.row_bytes <= p.piece_bytes) {
    p.rows_per_piece = static_cast<int32_t>(p.piece_bytes / p.row_bytes);
    p.segs_per_row = 1;
  } else {
    p.rows_per_piece = 0;
    p.segs_per_row = static_cast<int32_t>(cdiv64(p.row_bytes, p.piece_bytes));
  }
  auto pieces = [&](int64_t rows) -> int32_t {
    return p.rows_per_piece > 0 ? static_cast<int32_t>(cdiv64(rows, p.rows_per_piece))
                                : static_cast<int32_t>(rows * p.segs_per_row);
  };
  p.pieces_full = pieces(std::min<int64_t>(d.Cr, d.Ms));
  p.pieces_last = pieces(d.Ms - static_cast<int64_t>(d.nC - 1) * d.Cr);
  p.src_rows_contig = d.lda == d.K ? 1 : 0;
}

dt_status ag_common(const void* const* a_shards, const void* b, void* c, void* ws,
                    size_t ws_bytes, const dt_args* a, Derived* d) {
  dt_status s = derive(a, DT_OP_AG_GEMM, d);
  if (s != DT_OK) return s;
  if (!a_shards) return fail(DT_ERR_INVALID, "a_shards is NULL");
  if (d->M == 0 || d->N == 0) return DT_OK;
  for (int i = 0; i < d->W; ++i)
    if (!a_shards[i] || !is_aligned(a_shards[i], 16))
      return fail(DT_ERR_INVALID, "shard %d is NULL or not 16-byte aligned", i);
  if (!b || !is_aligned(b, 16) || !c || !is_aligned(c, 16))
    return fail(DT_ERR_INVALID, "B and C must be non-NULL and 16-byte aligned");
  return check_ws(*d, ws, ws_bytes);
}

// The own rank's block is tile-aligned (no tile straddles it): its tiles can read the shard
// in place and its chunks need no transfer.
bool own_in_place(const Derived& d) {
  if (d.W < 2) return false;
  const int64_t lo = static_cast<int64_t>(d.rank) * d.Ms, hi = lo + d.Ms;
  return lo % kBM == 0 && (hi % kBM == 0 || hi == d.M);
}

// copy chunk (s, j) of shard s into the gather buffer on `st`
dt_status ce_copy_chunk(const Derived& d, const void* const* a_shards, uint8_t* gather, int32_t s,
                        int32_t j, cudaStream_t st) {
  const int64_t r0 = static_cast<int64_t>(j) * d.Cr;
  const int64_t rows = std::min<int64_t>(d.Cr, d.Ms - r0);
  const uint8_t* src = reinterpret_cast<const uint8_t*>(a_shards[s]) + r0 * d.lda * 2;
  uint8_t* dst = gather + (static_cast<int64_t>(s) * d.Ms + r0) * d.ld_gather * 2;
  if (d.lda == d.K && d.ld_gather == d.K)  // rows back to back on both sides
    DT_CUDA(cudaMemcpyAsync(dst, src, static_cast<size_t>(rows * d.K * 2), cudaMemcpyDeviceToDevice, st));
  else
    DT_CUDA(cudaMemcpy2DAsync(dst, d.ld_gather * 2, src, d.lda * 2, d.K * 2, rows,
                              cudaMemcpyDeviceToDevice, st));
  return DT_OK;
}

}  // namespace

namespace dt {

void set_last_error(const char* msg) { g_last_error = msg; }

dt_status ag_gemm_on_scratch(const void* const* a_shards, const void* b, void* c, void* scratch,
                             size_t scratch_bytes, const dt_args* a, cudaStream_t stream) {
  g_last_error.clear();
  Derived d;
  dt_status s = ag_common(a_shards, b, c, scratch, scratch_bytes, a, &d);
  if (s != DT_OK || d.M == 0 || d.N == 0) return s;
  if (a->backend == DT_XFER_COPY_ENGINE || a->backend == DT_XFER_TMA_TILE)
    return fail(DT_ERR_UNSUPPORTED,
                "the fixed scratch runs the in-kernel transfer: use DT_XFER_TMA or DT_XFER_LDST");
  const int copy = a->backend == DT_XFER_LDST ? kCopyLdst : kCopyTma;
  if (d.K == 0) return launch_zero(c, d.M, d.N * (d.f32 ? 4 : 2), d.ldc * (d.f32 ? 4 : 2), stream);
  int dev = 0, sms = 0;
  DT_CUDA(cudaGetDevice(&dev));
  DT_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  uint8_t* w = reinterpret_cast<uint8_t*>(scratch);
  // start from a cleared error word and tag: the prepare kernel below then rewrites the order
  // and zeroes the flags and counters, whatever an earlier call left behind
  DT_CUDA(cudaMemsetAsync(w, 0, kTagOffset + sizeof(unsigned long long), stream));
  if ((s = launch_prepare(d, scratch, stream)) != DT_OK) return s;
  const uint32_t epoch = 1u;  // the flags were just zeroed
  KParams p;
  fill_common(p, d, scratch, epoch);
  for (int i = 0; i < d.W; ++i) p.shard[i] = reinterpret_cast<const uint8_t*>(a_shards[i]);
  p.out[0] = c;
  p.gather = w + d.off_data;
  p.ready = reinterpret_cast<uint32_t*>(w + d.off_ready);
  p.pieces_done = reinterpret_cast<uint32_t*>(w + d.off_pieces);
  p.lda_src = d.lda;
  p.ld_gather = d.ld_gather;
  p.wait_flags = 1;
  set_pieces(p, d, false);
  set_drop_chunk(p, d, take_drop_transfer());
  if ((s = make_tmap(&p.tmA[0], p.gather, d.K, d.M, d.ld_gather * 2, 64, kBM)) != DT_OK) return s;
  if ((s = make_tmap(&p.tmB[0], b, d.N, d.K, d.ldb * 2, 64, kBK)) != DT_OK) return s;
  p.own_in_place = own_in_place(d) ? 1 : 0;
  if (p.own_in_place &&
      (s = make_tmap(&p.tmA[1], a_shards[d.rank], d.K, d.Ms, d.lda * 2, 64, kBM)) != DT_OK)
    return s;
  const int use = a->num_sms > 0 ? std::min(a->num_sms, sms) : sms;
  if (d.copy_ctas >= use) return fail(DT_ERR_INVALID, "copy_ctas must leave SMs for the GEMM");
  p.copy_ctas = d.copy_ctas;
  const int grid = d.copy_ctas + grid_for(d, d.T, use - d.copy_ctas);
  const cudaError_t e = launch_ag_kernel(p, copy, d.f32, grid, true, stream, d.cl);
  if (e != cudaSuccess) return cuda_fail(e, "fused AllGather-GEMM launch");
  return DT_OK;
}

}  // namespace dt

// ================================================================================ C ABI
extern "C" {

void dt_args_default(dt_args* a) {
  if (!a) return;
  memset(a, 0, sizeof(*a));
  a->world_size = 1;
  a->swizzle = 1;
  a->backend = DT_XFER_AUTO;
  a->out_dtype = DT_BF16;
  a->tile_m = 0;  // CTA pairs when the problem has enough 256-row tiles
  a->tile_n = kBN;
  a->group = 8;
  a->chunk_rows = 128;
}

int dt_version(void) { return 300; }  // 3.0.0: dt_args.col_band, dt_tune_point carries col_band

size_t dt_sizeof_args(void) { return sizeof(dt_args); }
size_t dt_sizeof_tune_point(void) { return sizeof(dt_tune_point); }

const char* dt_status_string(dt_status s) {
  switch (s) {
    case DT_OK: return "DT_OK";
    case DT_ERR_INVALID: return "DT_ERR_INVALID";
    case DT_ERR_UNSUPPORTED: return "DT_ERR_UNSUPPORTED";
    case DT_ERR_TIMEOUT: return "DT_ERR_TIMEOUT";
    case DT_ERR_CUDA: return "DT_ERR_CUDA";
    case DT_ERR_WORKSPACE: return "DT_ERR_WORKSPACE";
  }
  return "DT_ERR_UNKNOWN";
}

const char* dt_last_error(void) { return g_last_error.c_str(); }

size_t dt_workspace_size(const dt_args* a, int op) {
  Derived d;
  if (derive(a, op, &d) != DT_OK) return 0;
  return d.total;
}

dt_status dt_workspace_init(const dt_args* a, int op, void* ws, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  Derived d;
  dt_status s = derive(a, op, &d);
  if (s != DT_OK) return s;
  s = check_ws(d, ws, ws_bytes);
  if (s != DT_OK) return s;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_ws.erase(ws);
  }
  DT_CUDA(cudaMemsetAsync(ws, 0, d.ctl_bytes, reinterpret_cast<cudaStream_t>(stream)));
  return DT_OK;
}

int64_t dt_tile_count(const dt_args* a, int op) {
  Derived d;
  if (derive(a, op, &d) != DT_OK) return -1;
  return d.T;
}

int32_t dt_tile_rows(const dt_args* a, int op) {
  Derived d;
  if (derive(a, op, &d) != DT_OK) return -1;
  return d.bm;
}

int32_t dt_col_band(const dt_args* a, int op) {
  Derived d;
  if (derive(a, op, &d) != DT_OK) return -1;
  return d.geom.Nb;
}

dt_status dt_swizzle_plan(const dt_args* a, int op, int32_t* order, int64_t len) {
  g_last_error.clear();
  Derived d;
  dt_status s = derive(a, op, &d);
  if (s != DT_OK) return s;
  if (len != d.T) return fail(DT_ERR_INVALID, "len %lld != tile count %d", (long long)len, d.T);
  if (d.T == 0) return DT_OK;
  if (!order) return fail(DT_ERR_INVALID, "order is NULL");
  std::vector<uint8_t> seen(d.T, 0);
  for (int32_t t = 0; t < d.T; ++t) {
    const int64_t pos = tile_position(d.geom, op, t);
    if (pos < 0 || pos >= d.T || seen[pos]) return fail(DT_ERR_INVALID, "plan is not a bijection");
    seen[pos] = 1;
    order[pos] = t;
  }
  return DT_OK;
}

dt_status dt_swizzle_plan_device(const dt_args* a, int op, int32_t* order_dev, int64_t len,
                                 void* stream) {
  g_last_error.clear();
  Derived d;
  dt_status s = derive(a, op, &d);
  if (s != DT_OK) return s;
  if (len != d.T) return fail(DT_ERR_INVALID, "len %lld != tile count %d", (long long)len, d.T);
  if (d.T == 0) return DT_OK;
  if (!order_dev) return fail(DT_ERR_INVALID, "order is NULL");
  plan_kernel<<<static_cast<unsigned>(cdiv64(d.T, 256)), 256, 0,
                reinterpret_cast<cudaStream_t>(stream)>>>(d.geom, op, order_dev, d.T);
  DT_CUDA(cudaGetLastError());
  return DT_OK;
}

dt_status dt_ag_gemm(const void* const* a_shards, const void* b, void* c, void* ws,
                     size_t ws_bytes, const dt_args* a, void* stream_) {
  NvtxRange range("dt_ag_gemm");
  g_last_error.clear();
  Derived d;
  dt_status s = ag_common(a_shards, b, c, ws, ws_bytes, a, &d);
  if (s != DT_OK || d.M == 0 || d.N == 0) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (d.K == 0) return launch_zero(c, d.M, d.N * (d.f32 ? 4 : 2), d.ldc * (d.f32 ? 4 : 2), stream);
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  uint32_t epoch = 0;
  if ((s = prepare_workspace(d, ws, stream, &epoch)) != DT_OK) return s;

  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  uint8_t* gather = w + d.off_data;
  KParams p;
  fill_common(p, d, ws, epoch);
  for (int i = 0; i < d.W; ++i) p.shard[i] = reinterpret_cast<const uint8_t*>(a_shards[i]);
  p.out[0] = c;
  p.gather = gather;
  p.ready = reinterpret_cast<uint32_t*>(w + d.off_ready);
  p.pieces_done = reinterpret_cast<uint32_t*>(w + d.off_pieces);
  p.lda_src = d.lda;
  p.ld_gather = d.ld_gather;
  p.wait_flags = 1;
  set_pieces(p, d, d.copy_ctas > 0);
  if ((s = make_tmap(&p.tmA[0], gather, d.K, d.M, d.ld_gather * 2, 64, kBM)) != DT_OK) return s;
  if ((s = make_tmap(&p.tmB[0], b, d.N, d.K, d.ldb * 2, 64, kBK)) != DT_OK) return s;
  p.own_in_place = own_in_place(d) ? 1 : 0;
  if (p.own_in_place &&
      (s = make_tmap(&p.tmA[1], a_shards[d.rank], d.K, d.Ms, d.lda * 2, 64, kBM)) != DT_OK)
    return s;
  if ((s = attach_trace(p, d, stream)) != DT_OK) return s;
  p.c_tma = c_tma_setting();
  if (p.c_tma && (s = make_c_tmap(&p.tmOut[0], c, d.M, d.N, d.ldc, d.f32)) != DT_OK) return s;

  const int sms = a->num_sms > 0 ? std::min(a->num_sms, dev->sms) : dev->sms;
  const int grid = grid_for(d, d.T, sms);
  if (d.W == 1) {
    // one rank gathers nothing: the GEMM reads its shard where it is
    if ((s = make_tmap(&p.tmA[0], a_shards[0], d.K, d.M, d.lda * 2, 64, kBM)) != DT_OK) return s;
    p.wait_flags = 0;
    cudaError_t e = launch_ag_kernel(p, kCopyNone, d.f32, grid, false, stream, d.cl);
    if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
    return DT_OK;
  }
  if (d.backend == DT_XFER_TMA_TILE) {
    // every tile loads its A rows from the owning shard (tmA[s]); no transfer, no flags
    for (int q = 0; q < d.W; ++q)
      if ((s = make_tmap(&p.tmA[q], a_shards[q], d.K, d.Ms, d.lda * 2, 64, kBM)) != DT_OK) return s;
    p.a_from_shards = 1;
    p.wait_flags = 0;
    p.own_in_place = 0;
    cudaError_t e = launch_ag_kernel(p, kCopyNone, d.f32, grid, false, stream, d.cl);
    if (e != cudaSuccess) return cuda_fail(e, "fused AllGather-GEMM launch");
    return DT_OK;
  }
  if (d.backend == DT_XFER_COPY_ENGINE) {
    PfnWriteValue32 wv = write_value32();
    if (!wv) return fail(DT_ERR_CUDA, "cuStreamWriteValue32 entry point unavailable");
    const int32_t drop = take_drop_transfer();
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if ((s = fork_copies(dev, stream)) != DT_OK) return s;
    const int32_t nchunks = d.W * d.nC;
    bool launched = false;
    int32_t queued = 0;  // chunks queued so far: chunk n goes to copy stream n % kCopyStreams
    for (int32_t tc = 0; tc < nchunks; ++tc) {
      // start the GEMM once the chunks its first tiles need are queued (at once when the own
      // rank's tiles read in place)
      if ((tc == d.nC || p.own_in_place) && !launched) {
        cudaError_t e = launch_ag_kernel(p, kCopyNone, d.f32, grid, false, stream, d.cl);
        if (e != cudaSuccess) return cuda_fail(e, "fused AllGather-GEMM launch");
        launched = true;
      }
      int32_t cs, cj;
      ag_transfer_chunk(d.geom, tc, cs, cj);
      if (p.own_in_place && cs == d.rank) continue;  // read in place
      if (tc == drop) continue;  // the message never arrives: its consumers time out
      cudaStream_t cst = dev->copy[queued++ % kCopyStreams];
      if ((s = ce_copy_chunk(d, a_shards, gather, cs, cj, cst)) != DT_OK) return s;
      // the chunk's flag, written by the copy's own stream once the copy is complete
      const CUdeviceptr flag =
          reinterpret_cast<CUdeviceptr>(p.ready + (static_cast<int64_t>(cs) * d.nC + cj));
      const CUresult r = wv(reinterpret_cast<CUstream>(cst), flag, epoch, 0);
      if (r != CUDA_SUCCESS) return fail(DT_ERR_CUDA, "cuStreamWriteValue32 failed (%d)", (int)r);
    }
    if (!launched) {
      cudaError_t e = launch_ag_kernel(p, kCopyNone, d.f32, grid, false, stream, d.cl);
      if (e != cudaSuccess) return cuda_fail(e, "fused AllGather-GEMM launch");
    }
    return join_copies(dev, stream);
  }
  const int copy = d.backend == DT_XFER_TMA ? kCopyTma : kCopyLdst;
  p.copy_ctas = d.copy_ctas;
  if (d.copy_ctas >= sms) return fail(DT_ERR_INVALID, "copy_ctas must leave SMs for the GEMM");
  set_drop_chunk(p, d, take_drop_transfer());
  const int grid_ded = d.copy_ctas + grid_for(d, d.T, sms - d.copy_ctas);
  cudaError_t e =
      launch_ag_kernel(p, copy, d.f32, d.copy_ctas ? grid_ded : grid, true, stream, d.cl);
  if (e != cudaSuccess) return cuda_fail(e, "fused AllGather-GEMM launch");
  return DT_OK;
}

dt_status dt_allgather(const void* const* a_shards, void* out, void* ws, size_t ws_bytes,
                       const dt_args* a, void* stream_) {
  NvtxRange range("dt_allgather");
  g_last_error.clear();
  if (!a) return fail(DT_ERR_INVALID, "args is NULL");
  // the GEMM's N, B and C play no part: the geometry is derived with a placeholder N
  dt_args x = *a;
  x.n = 8;
  x.ldb = 0;
  x.ldc = 0;
  x.out_dtype = DT_BF16;
  x.tile_m = 0;
  x.copy_ctas = 0;
  x.act = DT_ACT_NONE;
  const int64_t ldo = a->ldc ? a->ldc : a->k;
  if (a->backend == DT_XFER_AUTO && ldo != a->k) x.backend = DT_XFER_COPY_ENGINE;  // strided rows
  if (a->backend == DT_XFER_TMA_TILE)
    return fail(DT_ERR_INVALID, "DT_XFER_TMA_TILE moves tiles into shared memory, not an AllGather");
  Derived d;
  dt_status s = derive(&x, DT_OP_AG_GEMM, &d);
  if (s != DT_OK) return s;
  if (!a_shards) return fail(DT_ERR_INVALID, "a_shards is NULL");
  if (d.M == 0 || d.K == 0) return DT_OK;
  if (ldo < d.K || ldo % 8)
    return fail(DT_ERR_INVALID, "out's leading dimension (ldc) must be >= K and a multiple of 8");
  for (int i = 0; i < d.W; ++i)
    if (!a_shards[i] || !is_aligned(a_shards[i], 16))
      return fail(DT_ERR_INVALID, "shard %d is NULL or not 16-byte aligned", i);
  if (!out || !is_aligned(out, 16)) return fail(DT_ERR_INVALID, "out must be non-NULL and 16-byte aligned");
  if (d.backend != DT_XFER_COPY_ENGINE && ldo != d.K)
    return fail(DT_ERR_UNSUPPORTED,
                "the in-kernel transfers write rows back to back: out's leading dimension must be K");
  if ((s = check_ws(d, ws, ws_bytes)) != DT_OK) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* dst = reinterpret_cast<uint8_t*>(out);
  d.ld_gather = ldo;  // the copies land in `out`
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  if (d.backend == DT_XFER_COPY_ENGINE) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if ((s = fork_copies(dev, stream)) != DT_OK) return s;
    for (int32_t tc = 0; tc < d.W * d.nC; ++tc) {
      int32_t cs, cj;
      ag_transfer_chunk(d.geom, tc, cs, cj);
      if ((s = ce_copy_chunk(d, a_shards, dst, cs, cj, dev->copy[tc % kCopyStreams])) != DT_OK)
        return s;
    }
    return join_copies(dev, stream);
  }
  uint32_t epoch = 0;
  if ((s = prepare_workspace(d, ws, stream, &epoch)) != DT_OK) return s;
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  KParams p;
  fill_common(p, d, ws, epoch);
  if ((s = attach_trace(p, d, stream)) != DT_OK) return s;
  p.T = 0;  // no GEMM tiles: every CTA is a transfer CTA
  for (int i = 0; i < d.W; ++i) p.shard[i] = reinterpret_cast<const uint8_t*>(a_shards[i]);
  p.gather = dst;
  p.ready = reinterpret_cast<uint32_t*>(w + d.off_ready);
  p.pieces_done = reinterpret_cast<uint32_t*>(w + d.off_pieces);
  p.lda_src = d.lda;
  p.ld_gather = ldo;
  p.own_in_place = 0;  // the own shard is copied too
  set_pieces(p, d, true);  // every CTA is a transfer CTA
  // descriptors the kernel prefetches at start (unused without tiles)
  if ((s = make_tmap(&p.tmA[0], out, d.K, d.M, ldo * 2, 64, kBM)) != DT_OK) return s;
  p.tmB[0] = p.tmA[0];
  const int sms = a->num_sms > 0 ? std::min(a->num_sms, dev->sms) : dev->sms;
  p.copy_ctas = sms;
  const int copy = d.backend == DT_XFER_LDST ? kCopyLdst : kCopyTma;
  cudaError_t e = launch_ag_kernel(p, copy, false, sms, false, stream, 1);
  if (e != cudaSuccess) return cuda_fail(e, "AllGather launch");
  return DT_OK;
}

dt_status dt_ag_gemm_kernel_overlap(const void* const* a_shards, const void* b, void* c,
                                    void* ws, size_t ws_bytes, const dt_args* a, void* stream_) {
  NvtxRange range("dt_ag_gemm_kernel_overlap");
  g_last_error.clear();
  Derived d;
  dt_status s = ag_common(a_shards, b, c, ws, ws_bytes, a, &d);
  if (s != DT_OK || d.M == 0 || d.N == 0) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (d.K == 0) return launch_zero(c, d.M, d.N * (d.f32 ? 4 : 2), d.ldc * (d.f32 ? 4 : 2), stream);
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  uint8_t* gather = reinterpret_cast<uint8_t*>(ws) + d.off_data;
  KParams p;
  fill_common(p, d, ws, 0);
  p.tag = nullptr;  // the baseline does not use (or vouch for) the tile order
  p.out[0] = c;
  p.plain = 1;
  p.wait_flags = 0;
  if ((s = make_tmap(&p.tmA[0], gather, d.K, d.M, d.ld_gather * 2, 64, kBM)) != DT_OK) return s;
  if ((s = make_tmap(&p.tmB[0], b, d.N, d.K, d.ldb * 2, 64, kBK)) != DT_OK) return s;
  const int sms = a->num_sms > 0 ? std::min(a->num_sms, dev->sms) : dev->sms;
  const int32_t nchunks = d.W * d.nC;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  while (static_cast<int32_t>(dev->chunk_events.size()) < nchunks) {
    cudaEvent_t ev;
    DT_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    dev->chunk_events.push_back(ev);
  }
  DT_CUDA(cudaEventRecord(dev->ev_start, stream));
  DT_CUDA(cudaStreamWaitEvent(dev->side, dev->ev_start, 0));
  for (int32_t tc = 0; tc < nchunks; ++tc) {
    int32_t cs, cj;
    ag_transfer_chunk(d.geom, tc, cs, cj);
    if ((s = ce_copy_chunk(d, a_shards, gather, cs, cj, dev->side)) != DT_OK) return s;
    DT_CUDA(cudaEventRecord(dev->chunk_events[tc], dev->side));
    DT_CUDA(cudaStreamWaitEvent(stream, dev->chunk_events[tc], 0));
    // one launch of the same GEMM over this chunk's rows
    const int64_t lo = static_cast<int64_t>(cs) * d.Ms + static_cast<int64_t>(cj) * d.Cr;
    const int64_t hi = static_cast<int64_t>(cs) * d.Ms + std::min<int64_t>((cj + 1) * d.Cr, d.Ms);
    p.row_lo = lo;
    p.row_hi = hi;
    p.Tm = static_cast<int32_t>(cdiv64(hi - lo, d.bm));
    p.T = p.Tm * d.Tn;
    cudaError_t e = launch_ag_kernel(p, kCopyNone, d.f32, grid_for(d, p.T, sms), false, stream, d.cl);
    if (e != cudaSuccess) return cuda_fail(e, "per-chunk GEMM launch");
  }
  DT_CUDA(cudaEventRecord(dev->ev_done, dev->side));
  DT_CUDA(cudaStreamWaitEvent(stream, dev->ev_done, 0));
  return DT_OK;
}

// ------------------------------------------------------------------------------ ReduceScatter / AllReduce
static dt_status rs_common(const void* const* a_, const void* const* b_, void* const* out, void* ws,
                           size_t ws_bytes, const dt_args* a, int op, Derived* d) {
  dt_status s = derive(a, op, d);
  if (s != DT_OK) return s;
  if (!a_ || !b_ || !out) return fail(DT_ERR_INVALID, "a, b and out arrays must be non-NULL");
  if (d->M == 0 || d->N == 0) return DT_OK;
  for (int i = 0; i < d->W; ++i) {
    if (!a_[i] || !is_aligned(a_[i], 16) || !b_[i] || !is_aligned(b_[i], 16))
      return fail(DT_ERR_INVALID, "A_%d / B_%d NULL or not 16-byte aligned", i, i);
    if (!out[i] || !is_aligned(out[i], 16))
      return fail(DT_ERR_INVALID, "out_%d NULL or not 16-byte aligned", i);
  }
  return check_ws(*d, ws, ws_bytes);
}

// AllReduce: one output copy when every rank's pointer is the same buffer, else W
static int32_t ar_copies_of(const Derived& d, void* const* out) {
  for (int i = 1; i < d.W; ++i)
    if (out[i] != out[0]) return d.W;
  return 1;
}

static dt_status rs_params(KParams& p, const Derived& d, const void* const* a_,
                           const void* const* b_, void* const* out, void* ws, uint32_t epoch) {
  fill_common(p, d, ws, epoch);
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  p.recv = reinterpret_cast<float*>(w + d.off_data);
  p.unit_cnt = reinterpret_cast<uint32_t*>(w + d.off_cnt);
  p.pieces_max = d.pieces_max;
  p.ar_copies = d.op == DT_OP_GEMM_AR ? ar_copies_of(d, out) : 0;
  p.rot = rot_setting();
  // running sums [M][N] fp32 and park slots [W (W-1) Ms][N] fp32, moved in 32 x 128 boxes
  dt_status st = make_tmap(&p.tmAcc, p.recv, d.N, d.M, d.N * 4, 32, kBM, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
  if (st != DT_OK) return st;
  if (d.W > 1) {
    st = make_tmap(&p.tmPark, p.recv + static_cast<size_t>(d.M) * d.N, d.N,
                   static_cast<uint64_t>(d.W - 1) * d.M, d.N * 4, 32, kBM,
                   CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
    if (st != DT_OK) return st;
  } else {
    p.tmPark = p.tmAcc;  // one rank never parks
  }
  // the final sums go out as 32 x 128 boxes: bf16 boxes are dense 64-byte rows, fp32 boxes
  // keep the running sums' swizzled layout
  const CUtensorMapDataType odt =
      d.f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle oswz = d.f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  const uint64_t orow_bytes = static_cast<uint64_t>(d.ldc) * (d.f32 ? 4 : 2);
  const int nout = p.ar_copies > 0 ? p.ar_copies : d.W;
  for (int q = 0; q < nout; ++q) {
    const dt_status s = make_tmap(&p.tmOut[q], out[q], d.N, p.ar_copies > 0 ? d.M : d.Ms,
                                  orow_bytes, 32, kBM, odt, oswz);
    if (s != DT_OK) return s;
  }
  for (int q = 0; q < d.W; ++q) {
    p.out[q] = out[q];
    dt_status s = make_tmap(&p.tmA[q], a_[q], d.K, d.M, d.lda * 2, 64, kBM);
    if (s != DT_OK) return s;
    s = make_tmap(&p.tmB[q], b_[q], d.N, d.K, d.ldb * 2, 64, kBK);
    if (s != DT_OK) return s;
  }
  return DT_OK;
}

static dt_status zero_reduce_outputs(const Derived& d, void* const* out, cudaStream_t stream) {
  const int64_t eb = d.f32 ? 4 : 2;
  const bool ar = d.op == DT_OP_GEMM_AR;
  const int n = ar ? ar_copies_of(d, out) : d.W;
  for (int q = 0; q < n; ++q) {
    const dt_status s = launch_zero(out[q], ar ? d.M : d.Ms, d.N * eb, d.ldc * eb, stream);
    if (s != DT_OK) return s;
  }
  return DT_OK;
}

static dt_status reduce_fused(const void* const* a_, const void* const* b_, void* const* out,
                              void* ws, size_t ws_bytes, const dt_args* a, void* stream_, int op) {
  NvtxRange range(op == DT_OP_GEMM_RS ? "dt_gemm_rs" : "dt_gemm_ar");
  g_last_error.clear();
  Derived d;
  dt_status s = rs_common(a_, b_, out, ws, ws_bytes, a, op, &d);
  if (s != DT_OK || d.M == 0 || d.N == 0) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (d.K == 0) return zero_reduce_outputs(d, out, stream);
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  uint32_t epoch = 0;
  if ((s = prepare_workspace(d, ws, stream, &epoch)) != DT_OK) return s;
  KParams p;
  if ((s = rs_params(p, d, a_, b_, out, ws, epoch)) != DT_OK) return s;
  const int sms = a->num_sms > 0 ? std::min(a->num_sms, dev->sms) : dev->sms;
  cudaError_t e = launch_rs_kernel(p, d.f32, grid_for(d, d.T, sms), stream, d.cl);
  if (e != cudaSuccess) return cuda_fail(e, "fused GEMM-ReduceScatter / AllReduce launch");
  return DT_OK;
}

static dt_status reduce_kernel_overlap(const void* const* a_, const void* const* b_,
                                       void* const* out, void* ws, size_t ws_bytes,
                                       const dt_args* a, void* stream_, int op) {
  NvtxRange range(op == DT_OP_GEMM_RS ? "dt_gemm_rs_kernel_overlap" : "dt_gemm_ar_kernel_overlap");
  g_last_error.clear();
  Derived d;
  dt_status s = rs_common(a_, b_, out, ws, ws_bytes, a, op, &d);
  if (s != DT_OK || d.M == 0 || d.N == 0) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (d.K == 0) return zero_reduce_outputs(d, out, stream);
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  KParams p;
  if ((s = rs_params(p, d, a_, b_, out, ws, 0)) != DT_OK) return s;
  p.tag = nullptr;
  p.plain = 1;
  const bool ar = op == DT_OP_GEMM_AR;
  const int sms = a->num_sms > 0 ? std::min(a->num_sms, dev->sms) : dev->sms;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  while (static_cast<int32_t>(dev->chunk_events.size()) < d.W) {
    cudaEvent_t ev;
    DT_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    dev->chunk_events.push_back(ev);
  }
  const float* recv = p.recv;
  for (int32_t st = 0; st < d.W; ++st) {
    // one GEMM launch for destination block st (all W sources), fp32 partials only
    p.row_lo = static_cast<int64_t>(st) * d.Ms;
    p.row_hi = p.row_lo + d.Ms;
    p.Tm = static_cast<int32_t>(cdiv64(d.Ms, d.bm));
    p.T = d.W * p.Tm * d.Tn;
    cudaError_t e = launch_rs_kernel(p, d.f32, grid_for(d, p.T, sms), stream, d.cl);
    if (e != cudaSuccess) return cuda_fail(e, "per-destination GEMM launch");
    DT_CUDA(cudaEventRecord(dev->chunk_events[st], stream));
    DT_CUDA(cudaStreamWaitEvent(dev->side, dev->chunk_events[st], 0));
    // the reduction of block st runs on the second stream
    OutRows rows;
    memset(&rows, 0, sizeof(rows));
    if (ar) {
      rows.n = p.ar_copies;
      for (int c = 0; c < rows.n; ++c) rows.p[c] = out[c];
      rows.row0 = static_cast<int64_t>(st) * d.Ms;
    } else {
      rows.n = 1;
      rows.p[0] = out[st];
      rows.row0 = 0;
    }
    const int64_t work = d.Ms * (d.N / 4);
    const int rgrid = static_cast<int>(std::min<int64_t>(cdiv64(work, 256), 2 * sms));
    reduce_slots_kernel<<<rgrid, 256, 0, dev->side>>>(recv, d.W, d.Ms, d.N, st, rows, d.ldc,
                                                      d.f32 ? 1 : 0);
    DT_CUDA(cudaGetLastError());
  }
  DT_CUDA(cudaEventRecord(dev->ev_done, dev->side));
  DT_CUDA(cudaStreamWaitEvent(stream, dev->ev_done, 0));
  return DT_OK;
}

dt_status dt_gemm_rs(const void* const* a_, const void* const* b_, void* const* out, void* ws,
                     size_t ws_bytes, const dt_args* a, void* stream) {
  return reduce_fused(a_, b_, out, ws, ws_bytes, a, stream, DT_OP_GEMM_RS);
}

dt_status dt_gemm_ar(const void* const* a_, const void* const* b_, void* const* out, void* ws,
                     size_t ws_bytes, const dt_args* a, void* stream) {
  return reduce_fused(a_, b_, out, ws, ws_bytes, a, stream, DT_OP_GEMM_AR);
}

dt_status dt_gemm_rs_kernel_overlap(const void* const* a_, const void* const* b_, void* const* out,
                                    void* ws, size_t ws_bytes, const dt_args* a, void* stream) {
  return reduce_kernel_overlap(a_, b_, out, ws, ws_bytes, a, stream, DT_OP_GEMM_RS);
}

dt_status dt_gemm_ar_kernel_overlap(const void* const* a_, const void* const* b_, void* const* out,
                                    void* ws, size_t ws_bytes, const dt_args* a, void* stream) {
  return reduce_kernel_overlap(a_, b_, out, ws, ws_bytes, a, stream, DT_OP_GEMM_AR);
}

// ------------------------------------------------------------------------------ AllToAll
static dt_status a2a_common(const void* const* a_, const void* const* b_, void* const* out,
                            void* ws, size_t ws_bytes, const dt_args* a, Derived* d) {
  dt_status s = derive(a, DT_OP_GEMM_A2A, d);
  if (s != DT_OK) return s;
  if (!a_ || !b_ || !out) return fail(DT_ERR_INVALID, "a, b and out arrays must be non-NULL");
  if (d->M == 0 || d->N == 0) return DT_OK;
  for (int i = 0; i < d->W; ++i) {
    if (!a_[i] || !is_aligned(a_[i], 16) || !b_[i] || !is_aligned(b_[i], 16))
      return fail(DT_ERR_INVALID, "A_%d / B_%d NULL or not 16-byte aligned", i, i);
    if (!out[i] || !is_aligned(out[i], 16))
      return fail(DT_ERR_INVALID, "out_%d NULL or not 16-byte aligned", i);
  }
  return check_ws(*d, ws, ws_bytes);
}

static dt_status a2a_params(KParams& p, const Derived& d, const void* const* a_,
                            const void* const* b_, void* ws, uint32_t epoch) {
  fill_common(p, d, ws, epoch);
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  p.unit_cnt = reinterpret_cast<uint32_t*>(w + d.off_cnt);
  p.ready = reinterpret_cast<uint32_t*>(w + d.off_ready);
  p.row_hi = d.Ms;  // each rank's rows are tiled on their own
  p.a2a_step = -1;
  for (int q = 0; q < d.W; ++q) {
    dt_status s = make_tmap(&p.tmA[q], a_[q], d.K, d.Ms, d.lda * 2, 64, kBM);
    if (s != DT_OK) return s;
    s = make_tmap(&p.tmB[q], b_[q], d.N, d.K, d.ldb * 2, 64, kBK);
    if (s != DT_OK) return s;
  }
  return DT_OK;
}

static dt_status zero_a2a_outputs(const Derived& d, void* const* out, cudaStream_t stream) {
  const int64_t eb = d.f32 ? 4 : 2;
  for (int h = 0; h < d.W; ++h) {
    const dt_status s = launch_zero(out[h], d.M, d.geom.Nw * eb, d.ldc * eb, stream);
    if (s != DT_OK) return s;
  }
  return DT_OK;
}

dt_status dt_gemm_a2a(const void* const* a_, const void* const* b_, void* const* out, void* ws,
                      size_t ws_bytes, const dt_args* a, void* stream_) {
  NvtxRange range("dt_gemm_a2a");
  g_last_error.clear();
  Derived d;
  dt_status s = a2a_common(a_, b_, out, ws, ws_bytes, a, &d);
  if (s != DT_OK || d.M == 0 || d.N == 0) return s;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (d.K == 0) return zero_a2a_outputs(d, out, stream);
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  uint32_t epoch = 0;
  if ((s = prepare_workspace(d, ws, stream, &epoch)) != DT_OK) return s;
  KParams p;
  if ((s = a2a_params(p, d, a_, b_, ws, epoch)) != DT_OK) return s;
  for (int h = 0; h < d.W; ++h) p.out[h] = out[h];
  p.c_tma = c_tma_setting();
  for (int h = 0; h < d.W && p.c_tma; ++h)
    if ((s = make_a2a_out_tmap(&p.tmOut[h], out[h], d.Ms, d.geom.Nw, d.ldc, d.W, d.f32)) != DT_OK)
      return s;
  const int sms = a->num_sms > 0 ? std::min(a->num_sms, dev->sms) : dev->sms;
  cudaError_t e = launch_a2a_kernel(p, d.f32, grid_for(d, d.T, sms), stream, d.cl);
  if (e != cudaSuccess) return cuda_fail(e, "fused GEMM-AllToAll launch");
  return DT_OK;
}

dt_status dt_gemm_a2a_kernel_overlap(const void* const* a_, const void* const* b_,
                                     void* const* y, void* const* out, void* ws, size_t ws_bytes,
                                     const dt_args* a, void* stream_) {
  NvtxRange range("dt_gemm_a2a_kernel_overlap");
  g_last_error.clear();
  Derived d;
  dt_status s = a2a_common(a_, b_, out, ws, ws_bytes, a, &d);
  if (s != DT_OK || d.M == 0 || d.N == 0) return s;
  if (!y) return fail(DT_ERR_INVALID, "y array must be non-NULL");
  for (int q = 0; q < d.W; ++q)
    if (!y[q] || !is_aligned(y[q], 16)) return fail(DT_ERR_INVALID, "y_%d NULL or not 16-byte aligned", q);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (d.K == 0) return zero_a2a_outputs(d, out, stream);
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  KParams p;
  if ((s = a2a_params(p, d, a_, b_, ws, 0)) != DT_OK) return s;
  p.tag = nullptr;
  p.plain = 1;
  p.ldc = d.N;  // the ranks' own Y_q
  for (int q = 0; q < d.W; ++q) p.out[q] = y[q];
  p.T = d.W * d.Tm * d.geom.Tnw;
  const int eb = d.f32 ? 4 : 2;
  const int sms = a->num_sms > 0 ? std::min(a->num_sms, dev->sms) : dev->sms;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  while (static_cast<int32_t>(dev->chunk_events.size()) < d.W) {
    cudaEvent_t ev;
    DT_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    dev->chunk_events.push_back(ev);
  }
  for (int32_t st = 0; st < d.W; ++st) {
    // step st: every rank q computes the block of destination (q + st + 1) mod W
    p.a2a_step = st;
    cudaError_t e = launch_a2a_kernel(p, d.f32, grid_for(d, p.T, sms), stream, d.cl);
    if (e != cudaSuccess) return cuda_fail(e, "per-step GEMM launch");
    DT_CUDA(cudaEventRecord(dev->chunk_events[st], stream));
    DT_CUDA(cudaStreamWaitEvent(dev->side, dev->chunk_events[st], 0));
    // the all-to-all of this step on the copy engine, overlapping the next step's GEMM
    for (int32_t q = 0; q < d.W; ++q) {
      const int32_t h = (q + st + 1) % d.W;
      const uint8_t* src = reinterpret_cast<const uint8_t*>(y[q]) + h * d.geom.Nw * eb;
      uint8_t* dst = reinterpret_cast<uint8_t*>(out[h]) + static_cast<size_t>(q) * d.Ms * d.ldc * eb;
      DT_CUDA(cudaMemcpy2DAsync(dst, d.ldc * eb, src, d.N * eb, d.geom.Nw * eb, d.Ms,
                                cudaMemcpyDeviceToDevice, dev->side));
    }
  }
  DT_CUDA(cudaEventRecord(dev->ev_done, dev->side));
  DT_CUDA(cudaStreamWaitEvent(stream, dev->ev_done, 0));
  return DT_OK;
}

dt_status dt_a2a_signals(const dt_args* a, void* ws, void* stream_, uint32_t* flags,
                         uint32_t* counts, int64_t len, uint32_t* epoch) {
  g_last_error.clear();
  Derived d;
  dt_status s = derive(a, DT_OP_GEMM_A2A, &d);
  if (s != DT_OK) return s;
  const int64_t n = static_cast<int64_t>(d.W) * d.W * d.nC;
  if (len != n) return fail(DT_ERR_INVALID, "len %lld != W*W*nC = %lld", (long long)len, (long long)n);
  if (!ws) return fail(DT_ERR_WORKSPACE, "workspace is NULL");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  DT_CUDA(cudaStreamSynchronize(stream));
  const uint8_t* w = reinterpret_cast<const uint8_t*>(ws);
  if (flags && n > 0) DT_CUDA(cudaMemcpy(flags, w + d.off_ready, 4 * n, cudaMemcpyDeviceToHost));
  if (counts && n > 0) DT_CUDA(cudaMemcpy(counts, w + d.off_cnt, 4 * n, cudaMemcpyDeviceToHost));
  if (epoch) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_ws.find(ws);
    *epoch = it == g_ws.end() ? 0u : it->second.epoch;
  }
  return DT_OK;
}

// ------------------------------------------------------------------------------ tuner
}  // extern "C"

namespace {

struct TuneCtx {
  cudaStream_t stream;
  void* ws;
  size_t ws_bytes;
  int32_t reps;
  cudaEvent_t t0, t1;
};

// Time one candidate: one warm-up call, then `reps` calls between two events.
template <typename Call>
void tune_one(const TuneCtx& t, dt_args& cand, int op, Call&& call, dt_tune_point* pt) {
  pt->chunk_rows = cand.chunk_rows;
  pt->backend = cand.backend;
  pt->copy_ctas = cand.copy_ctas;
  pt->swizzle = cand.swizzle;
  pt->group = cand.group;
  pt->tile_m = cand.tile_m;
  pt->col_band = cand.col_band;
  pt->ms = -1.0f;
  const size_t need = dt_workspace_size(&cand, op);
  if (need == 0 || need > t.ws_bytes) {
    pt->status = need == 0 ? DT_ERR_INVALID : DT_ERR_WORKSPACE;
    return;
  }
  dt_status st = call(cand);
  if (st == DT_OK) st = dt_check(t.ws, t.stream, nullptr);
  if (st != DT_OK) {
    pt->status = st;
    return;
  }
  cudaEventRecord(t.t0, t.stream);
  for (int32_t r = 0; r < t.reps && st == DT_OK; ++r) st = call(cand);
  cudaEventRecord(t.t1, t.stream);
  if (st == DT_OK) st = dt_check(t.ws, t.stream, nullptr);
  float ms = 0.f;
  if (st == DT_OK && cudaEventElapsedTime(&ms, t.t0, t.t1) == cudaSuccess) pt->ms = ms / t.reps;
  pt->status = st;
}

// Under the power cap the GPU's clock drifts as it warms, which would favour whatever is timed
// first.  A forward pass times every candidate and picks the fastest as the reference; a
// reverse pass then times each candidate between two timings of the reference and scores it
// by its time over the mean of those two, which cancels the drift.  A point's reported time is
// its score times the median of the reference's timings.
template <typename Call>
std::vector<dt_tune_point> tune_all(const TuneCtx& t, std::vector<dt_args>& cands, int op,
                                    Call&& call) {
  std::vector<dt_tune_point> pts(cands.size());
  const int n = static_cast<int>(cands.size());
  int ref = -1;
  for (int i = 0; i < n; ++i) {
    tune_one(t, cands[i], op, call, &pts[i]);
    if (pts[i].status == DT_OK && pts[i].ms >= 0 && (ref < 0 || pts[i].ms < pts[ref].ms)) ref = i;
  }
  if (ref < 0 || n < 2) return pts;
  std::vector<float> ref_ms;
  auto time_ref = [&]() -> float {
    dt_tune_point r;
    tune_one(t, cands[ref], op, call, &r);
    if (r.status == DT_OK && r.ms > 0) ref_ms.push_back(r.ms);
    return r.status == DT_OK ? r.ms : -1.0f;
  };
  std::vector<float> score(n, -1.0f);
  score[ref] = 1.0f;
  float before = time_ref();
  for (int i = n - 1; i >= 0 && before > 0; --i) {
    if (i == ref || pts[i].status != DT_OK) continue;
    dt_tune_point again;
    tune_one(t, cands[i], op, call, &again);
    const float after = time_ref();
    if (again.status != DT_OK) {
      pts[i] = again;
    } else if (after > 0 && again.ms >= 0) {
      score[i] = again.ms / (0.5f * (before + after));
    }
    if (after <= 0) break;
    before = after;
  }
  if (ref_ms.empty()) return pts;
  std::sort(ref_ms.begin(), ref_ms.end());
  const float ref_med = ref_ms[ref_ms.size() / 2];
  for (int i = 0; i < n; ++i)
    if (pts[i].status == DT_OK && score[i] > 0) pts[i].ms = score[i] * ref_med;
  return pts;
}

std::vector<int64_t> chunk_candidates(int64_t ms) {
  std::vector<int64_t> v;
  for (int64_t c : {64, 128, 256, 512, 1024, 2048, 4096})
    if (c < ms) v.push_back(c);
  v.push_back(std::max<int64_t>(ms, 1));
  return v;
}

dt_status tune_setup(int op, const dt_args* a, void* ws, size_t ws_bytes, int32_t reps,
                     void* stream, TuneCtx* t, Derived* d) {
  dt_status s = derive(a, op, d);
  if (s != DT_OK) return s;
  if (reps < 1) return fail(DT_ERR_INVALID, "reps must be >= 1");
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!dev->tune_t0) {
      DT_CUDA(cudaEventCreate(&dev->tune_t0));
      DT_CUDA(cudaEventCreate(&dev->tune_t1));
    }
  }
  *t = TuneCtx{reinterpret_cast<cudaStream_t>(stream), ws, ws_bytes, reps, dev->tune_t0,
               dev->tune_t1};
  return DT_OK;
}

// A 64-bit hash of the tile order `a` gives for `op` (0 if `a` is invalid).
uint64_t order_hash(const dt_args& a, int op) {
  Derived d;
  if (derive(&a, op, &d) != DT_OK) return 0;
  uint64_t h = 1469598103934665603ull;
  for (int32_t t = 0; t < d.T; ++t) {
    h ^= static_cast<uint64_t>(tile_position(d.geom, op, t));
    h *= 1099511628211ull;
  }
  return h;
}

// Drop candidates that would run exactly the same kernel as an earlier one: same chunk rows,
// tile rows and transfer, and a group width or column band that yields the same tile order
// (a group at least as wide as every key's m-tiles, a band as wide as all column tiles).
void drop_same_order(std::vector<dt_args>& cands, int op) {
  std::vector<dt_args> keep;
  std::vector<uint64_t> hashes;
  for (const dt_args& c : cands) {
    const uint64_t h = order_hash(c, op);
    bool dup = false;
    for (size_t k = 0; k < keep.size() && !dup; ++k)
      dup = h != 0 && h == hashes[k] && keep[k].chunk_rows == c.chunk_rows &&
            keep[k].tile_m == c.tile_m && keep[k].backend == c.backend &&
            keep[k].copy_ctas == c.copy_ctas;
    if (!dup) {
      keep.push_back(c);
      hashes.push_back(h);
    }
  }
  cands.swap(keep);
}

// Pick the point to keep and copy its knobs into *a.  The tuner times short bursts at full
// clock; run for longer under the power cap, a kernel's clock follows its energy, so among
// near-equal points the one that moves the fewest DRAM bytes is kept.
// * Reduce ops: automatic column bands (they keep B_q's band in L2: the FFN pair's
//   ReduceScatter reads 3.9-4.9 GB per launch with two bands against 5.3-5.9 GB with one) are
//   kept unless one band is more than kBandTie faster in the burst: in the timed steps of the
//   benchmark, after the tuner, two bands took 2.06-2.11 ms and one band 2.17-2.21 ms on the
//   same boxes, while the tuner's bursts had put one band up to ~1 % ahead.
// * Then, among the points within kTuneTie of the fastest (of the kept bands), the largest
//   chunk rows, then the fastest.  Fewer, larger chunks mean fewer key groups in the order, each
//   of which re-streams B from DRAM (the largest AllGather with the per-tile pull, 3 s runs:
//   chunk 2048 / 1024 / 256 read 2.52 / 3.06 / 4.28 GB per launch and took 1.282 / 1.315 /
//   1.343 ms at 1425 / 1387 / 1350-1365 MHz, where their burst times lie within 1 %).  The
//   AllGather's column bands move more bytes at some chunk sizes and fewer at others, so they
//   are measured, not ranked.
constexpr float kTuneTie = 1.01f;
constexpr float kBandTie = 1.04f;
dt_status tune_finish(std::vector<dt_tune_point>& pts, dt_args* a, dt_tune_point* out,
                      int32_t max_points, int32_t* n_points, bool bands_first) {
  auto ran = [&](const dt_tune_point& x) { return x.status == DT_OK && x.ms >= 0; };
  int fastest = -1;
  for (int i = 0; i < static_cast<int>(pts.size()); ++i)
    if (ran(pts[i]) && (fastest < 0 || pts[i].ms < pts[fastest].ms)) fastest = i;
  // reduce ops: stay with the automatic bands when their best point is within kBandTie
  bool auto_only = false;
  if (bands_first && fastest >= 0 && pts[fastest].col_band != 0) {
    int best_auto = -1;
    for (int i = 0; i < static_cast<int>(pts.size()); ++i)
      if (ran(pts[i]) && pts[i].col_band == 0 && (best_auto < 0 || pts[i].ms < pts[best_auto].ms))
        best_auto = i;
    if (best_auto >= 0 && pts[best_auto].ms <= kBandTie * pts[fastest].ms) {
      fastest = best_auto;
      auto_only = true;
    }
  }
  int best = fastest;
  auto larger_chunk = [&](const dt_tune_point& x, const dt_tune_point& y) {
    if (x.chunk_rows != y.chunk_rows) return x.chunk_rows > y.chunk_rows;
    return x.ms < y.ms;
  };
  for (int i = 0; fastest >= 0 && i < static_cast<int>(pts.size()); ++i) {
    if (!ran(pts[i]) || pts[i].ms > kTuneTie * pts[fastest].ms) continue;
    if (auto_only && pts[i].col_band != 0) continue;
    if (bands_first && !auto_only && (pts[i].col_band == 0) != (pts[best].col_band == 0)) {
      if (pts[i].col_band == 0) best = i;  // automatic bands before one band
      continue;
    }
    if (larger_chunk(pts[i], pts[best])) best = i;
  }
  if (n_points) *n_points = static_cast<int32_t>(pts.size());
  if (out)
    for (int i = 0; i < static_cast<int>(pts.size()) && i < max_points; ++i) out[i] = pts[i];
  if (best < 0) return fail(DT_ERR_UNSUPPORTED, "no tuner candidate ran");
  a->chunk_rows = pts[best].chunk_rows;
  a->backend = pts[best].backend;
  a->copy_ctas = pts[best].copy_ctas;
  a->swizzle = pts[best].swizzle;
  a->group = pts[best].group;
  a->tile_m = pts[best].tile_m;
  a->col_band = pts[best].col_band;
  return DT_OK;
}

}  // namespace

extern "C" {

dt_status dt_tune_ag_gemm(const void* const* a_shards, const void* b, void* c, void* ws,
                          size_t ws_bytes, dt_args* a, int32_t reps, dt_tune_point* points,
                          int32_t max_points, int32_t* n_points, void* stream) {
  g_last_error.clear();
  TuneCtx t;
  Derived d;
  dt_status s = tune_setup(DT_OP_AG_GEMM, a, ws, ws_bytes, reps, stream, &t, &d);
  if (s != DT_OK) return s;
  DevCtx* dev = nullptr;
  if ((s = dev_ctx(&dev)) != DT_OK) return s;
  auto call = [&](dt_args& cand) { return dt_ag_gemm(a_shards, b, c, ws, ws_bytes, &cand, stream); };
  // column bands: as given, and one band when that differs
  std::vector<int32_t> bands = {a->col_band};
  if (d.geom.Nb < d.Tn) bands.push_back(d.Tn);
  std::vector<dt_args> cands;
  for (int64_t cr : chunk_candidates(d.Ms)) {
    const int64_t nchunks = d.W * cdiv64(d.Ms, cr);
    struct V { int be; int copy; };
    std::vector<V> vs = {{DT_XFER_TMA, 0}, {DT_XFER_LDST, 0}};
    if (nchunks <= 512) vs.push_back({DT_XFER_COPY_ENGINE, 0});
    for (int n : {8, 16})
      if (dev->sms > 4 * n) {
        vs.push_back({DT_XFER_TMA, n});
        vs.push_back({DT_XFER_LDST, n});
      }
    if (d.Ms % kBM == 0) vs.push_back({DT_XFER_TMA_TILE, 0});  // per-tile pull, co-located
    for (const V& v : vs) {
      for (int32_t nb : bands) {
        dt_args cand = *a;
        cand.chunk_rows = cr;
        cand.backend = v.be;
        cand.copy_ctas = v.copy;
        cand.swizzle = 1;
        cand.group = a->group > 0 ? a->group : 8;
        cand.col_band = nb;
        cands.push_back(cand);
      }
    }
  }
  std::vector<dt_tune_point> pts = tune_all(t, cands, DT_OP_AG_GEMM, call);
  // tile order inside a chunk: group widths around the best point
  int best = -1;
  for (int i = 0; i < static_cast<int>(pts.size()); ++i)
    if (pts[i].status == DT_OK && pts[i].ms >= 0 && (best < 0 || pts[i].ms < pts[best].ms)) best = i;
  if (best >= 0) {
    const dt_tune_point base = pts[best];
    std::vector<dt_args> gc;
    for (int g : {4, 8, 16}) {
      dt_args cand = *a;
      cand.chunk_rows = base.chunk_rows;
      cand.backend = base.backend;
      cand.copy_ctas = base.copy_ctas;
      cand.col_band = base.col_band;
      cand.swizzle = 1;
      cand.group = g;
      gc.push_back(cand);
    }
    // the best point is timed again beside its group variants (those giving another order)
    drop_same_order(gc, DT_OP_AG_GEMM);
    if (gc.size() > 1)
      for (const dt_tune_point& pt : tune_all(t, gc, DT_OP_AG_GEMM, call)) pts.push_back(pt);
  }
  return tune_finish(pts, a, points, max_points, n_points, false);
}

dt_status dt_tune_reduce(int op, const void* const* a_, const void* const* b_, void* const* out,
                         void* ws, size_t ws_bytes, dt_args* a, int32_t reps, dt_tune_point* points,
                         int32_t max_points, int32_t* n_points, void* stream) {
  g_last_error.clear();
  if (op != DT_OP_GEMM_RS && op != DT_OP_GEMM_AR && op != DT_OP_GEMM_A2A)
    return fail(DT_ERR_INVALID, "dt_tune_reduce takes DT_OP_GEMM_RS, DT_OP_GEMM_AR or DT_OP_GEMM_A2A");
  TuneCtx t;
  Derived d;
  dt_status s = tune_setup(op, a, ws, ws_bytes, reps, stream, &t, &d);
  if (s != DT_OK) return s;
  auto call = [&](dt_args& cand) {
    if (op == DT_OP_GEMM_A2A) return dt_gemm_a2a(a_, b_, out, ws, ws_bytes, &cand, stream);
    return op == DT_OP_GEMM_RS ? dt_gemm_rs(a_, b_, out, ws, ws_bytes, &cand, stream)
                               : dt_gemm_ar(a_, b_, out, ws, ws_bytes, &cand, stream);
  };
  // column bands (ReduceScatter / AllReduce): as given, and one band when that differs
  std::vector<int32_t> bands = {a->col_band};
  if (op != DT_OP_GEMM_A2A && d.geom.Nb < d.Tn) bands.push_back(d.Tn);
  std::vector<dt_args> cands;
  for (int32_t nb : bands) {
    for (int64_t cr : chunk_candidates(d.Ms)) {
      for (int g : {4, 8, 16}) {
        dt_args cand = *a;
        cand.chunk_rows = cr;
        cand.swizzle = 1;
        cand.group = g;
        cand.col_band = nb;
        cands.push_back(cand);
      }
    }
  }
  drop_same_order(cands, op);
  std::vector<dt_tune_point> pts = tune_all(t, cands, op, call);
  return tune_finish(pts, a, points, max_points, n_points, true);
}

dt_status dt_ffn_ag_rs(const void* const* x_shards, const void* w1, const void* const* w2,
                       void* h, void* const* out, void* ws_ag, size_t ws_ag_bytes, void* ws_rs,
                       size_t ws_rs_bytes, const dt_args* ag, const dt_args* rs, void* stream) {
  g_last_error.clear();
  if (!ag || !rs || !w2 || !out) return fail(DT_ERR_INVALID, "NULL argument");
  const int32_t W = ag->world_size;
  if (rs->world_size != W || ag->m != rs->m || ag->n != static_cast<int64_t>(W) * rs->k)
    return fail(DT_ERR_INVALID, "the two GEMMs do not chain: need equal W and M, ag.n == W * rs.k");
  if (rs->k % 8) return fail(DT_ERR_UNSUPPORTED, "F per rank must be a multiple of 8");
  if (ag->out_dtype != DT_BF16 || (ag->ldc != 0 && ag->ldc != ag->n))
    return fail(DT_ERR_INVALID, "h must be bf16 with ldc == ag.n");
  if ((rs->lda != 0 && rs->lda != ag->n))
    return fail(DT_ERR_INVALID, "rs.lda must be ag.n (the row stride of h)");
  if (W < 1 || W > DT_MAX_WORLD) return fail(DT_ERR_INVALID, "world_size out of range");
  dt_status s = dt_ag_gemm(x_shards, w1, h, ws_ag, ws_ag_bytes, ag, stream);
  if (s != DT_OK) return s;
  dt_args r = *rs;
  r.lda = ag->n;
  const void* a_blocks[DT_MAX_WORLD];
  for (int q = 0; q < W; ++q)
    a_blocks[q] = reinterpret_cast<const uint8_t*>(h) + static_cast<size_t>(q) * rs->k * 2;
  return dt_gemm_rs(a_blocks, w2, out, ws_rs, ws_rs_bytes, &r, stream);
}

size_t dt_trace_bytes(const dt_args* a) {
  Derived d;
  if (derive(a, DT_OP_AG_GEMM, &d) != DT_OK) return 0;
  return trace_bytes_for(d.W, d.nC);
}

dt_status dt_trace_attach(void* trace, size_t bytes) {
  g_last_error.clear();
  if (trace != nullptr && !is_aligned(trace, 8)) return fail(DT_ERR_INVALID, "trace must be 8-byte aligned");
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace = trace;
  g_trace_bytes = trace ? bytes : 0;
  return DT_OK;
}

dt_status dt_debug_drop_transfer(int32_t step) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  g_drop_transfer = step;
  return DT_OK;
}

dt_status dt_check(void* ws, void* stream_, uint32_t* info) {
  g_last_error.clear();
  if (!ws) return fail(DT_ERR_WORKSPACE, "workspace is NULL");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  DT_CUDA(cudaStreamSynchronize(stream));
  uint32_t h[4] = {0, 0, 0, 0};
  DT_CUDA(cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost));
  if (info) memcpy(info, h, sizeof(h));
  if (h[0] == kDevOk) return DT_OK;
  // clear the error and the layout tag: the next call re-initialises the counters and flags
  // that the failed call may have left behind
  DT_CUDA(cudaMemset(ws, 0, kTagOffset + sizeof(unsigned long long)));
  if (h[0] == kDevBadTile)
    return fail(DT_ERR_INVALID, "device: tile id out of range at position %u", h[1]);
  return fail(DT_ERR_TIMEOUT, "device: bounded wait ran out (code %u, site %u, cta %u, %u)", h[0],
              h[1], h[2], h[3]);
}

}  // extern "C"
