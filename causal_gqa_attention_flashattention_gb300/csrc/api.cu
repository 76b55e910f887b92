// C-ABI layer of libneattn: argument checks, TMA descriptors, the rotary
// cos/sin table cache, the device status word, and kernel launches.
// The operations are defined in include/ne_attn.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/ne_attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace ne {

// ------------------------------------------------------------------ device status word
__device__ int g_status_word;

// ------------------------------------------------------------------ fixed scratch for ne_attn_bwd_noalloc
// Every GPU that loads this library holds this array until the process exits.
// Host code must not use the symbol as an address: ne_attn_bwd_noalloc asks
// the runtime for its device address (cudaGetSymbolAddress) once per device.
static __device__ __align__(256) unsigned char g_static_scratch[NE_ATTN_STATIC_SCRATCH_BYTES];

// ------------------------------------------------------------------ small kernels
// cos/sin of t * theta_i in double precision, rounded to fp32.
__global__ void k_rope_table(float2* tab, int Tcap, int D, double log2_base) {
  const int half = D / 2;
  const long long n = (long long)Tcap * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / half), i = (int)(idx % half);
    const double theta = exp2(-2.0 * (double)i / (double)D * log2_base);
    double s, c;
    sincos((double)t * theta, &s, &c);
    tab[idx] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_rope_table(float2* tab, int Tcap, int D, double base, cudaStream_t s) {
  const long long n = (long long)Tcap * (D / 2);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  k_rope_table<<<blocks, 256, 0, s>>>(tab, Tcap, D, std::log2(base));
  return cudaGetLastError();
}

__global__ void k_timeout_probe(int* status, long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing arrives on `bar`: the wait must give up after limit_ns.
    if (!mbar_wait(&bar, 0, &abort_flag, (unsigned long long)limit_ns)) atomicCAS(status, 0, kStatusTimeout);
  }
}

cudaError_t launch_timeout_probe(int* status, long long limit_ns, cudaStream_t s) {
  k_timeout_probe<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ per-device state
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

struct RopeTable {
  int D;
  double base;
  int Tcap;
  float2* ptr;
};

// Work items of the persistent forward, per CTA: see fwd_pair_schedule.
struct FwdSchedule {
  int B, Hkv, G, nt, nsm, grid, K;
  int* ptr;  // [grid, K] int4 entries, device
};

// Library-owned forward workspace of one stream (calls that pass none).
struct FwdScratch {
  cudaStream_t stream;
  void* ptr;
  size_t bytes;
};

struct DeviceState {
  bool init = false;
  bool supported = false;
  int* status = nullptr;
  std::vector<RopeTable> tables;
  std::vector<FwdSchedule> scheds;
  std::vector<FwdScratch> fwd_scratch;
  unsigned char* static_scratch = nullptr;  // device address of g_static_scratch (set on first use)
};

std::mutex g_mu;
DeviceState g_dev[64];
EncodeTiledFn g_encode = nullptr;

int current_device(int* dev) { return cudaGetDevice(dev) == cudaSuccess ? NE_OK : NE_ERR_CUDA; }

// Requires g_mu held.
int device_state(int dev, DeviceState** out) {
  if (dev < 0 || dev >= 64) return NE_ERR_UNSUPPORTED;
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return NE_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return NE_ERR_CUDA;
      d.status = static_cast<int*>(p);
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return NE_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.init = true;
  }
  if (!d.supported) return NE_ERR_UNSUPPORTED;
  *out = &d;
  return NE_OK;
}

// Returns a table with at least Tneed rows for (D, base) on this device.
// Requires g_mu held.
int rope_table(DeviceState& d, int D, double base, int Tneed, cudaStream_t s, const float2** out) {
  for (auto& t : d.tables)
    if (t.D == D && t.base == base && t.Tcap >= Tneed) {
      *out = t.ptr;
      return NE_OK;
    }
  int Tcap = ((Tneed + 1023) / 1024) * 1024;
  float2* p = nullptr;
  if (cudaMalloc(&p, sizeof(float2) * (size_t)Tcap * (D / 2)) != cudaSuccess) return NE_ERR_CUDA;
  if (launch_rope_table(p, Tcap, D, base, s) != cudaSuccess) {
    cudaFree(p);
    return NE_ERR_CUDA;
  }
  // Older, smaller tables stay allocated: kernels queued on other streams may still read them.
  d.tables.push_back(RopeTable{D, base, Tcap, p});
  *out = p;
  return NE_OK;
}

// The persistent forward's work items, built on the host once per shape.  A
// unit is one query head's 128-row query tile; an item pairs two units of one
// (batch, key/value head), which share its K/V stream (key tiles
// 0 .. max(i0, i1)), one softmax warpgroup per unit.  Pairs: heads 2k and 2k+1
// of the group at the same query tile; with an odd group size the last head of
// the group pairs its own adjacent tiles (nt-1, nt-2), (nt-3, nt-4), ..., and a
// leftover tile 0 goes alone.  An item costs 2 per unit key tile plus 1 per
// unit epilogue; items in decreasing cost (ties: larger tile, then batch, then
// key/value head, so a group's items go out together and meet in L2) each go
// to the CTA with the least work so far.  Entries are int4
// (b, h0 | (h1 + 1) << 16, i0, i1) with i0 >= i1 (h1 + 1 = 0: one unit);
// rows are padded with b = -1.  grid = min(items, nsm).
struct PairItem {
  int b, kvh, h0, h1, i0, i1;
  long long cost;
};
std::vector<int> fwd_pair_schedule(int B, int Hkv, int G, int nt, int nsm, int* grid_out, int* K) {
  std::vector<PairItem> items;
  for (int b = 0; b < B; b++)
    for (int g = 0; g < Hkv; g++) {
      const int h = g * G;
      for (int i = nt - 1; i >= 0; i--)
        for (int k = 0; k + 1 < G; k += 2) items.push_back(PairItem{b, g, h + k, h + k + 1, i, i, 0});
      if (G % 2 == 1)
        for (int i = nt - 1; i >= 0; i -= 2)
          items.push_back(PairItem{b, g, h + G - 1, i >= 1 ? h + G - 1 : -1, i, i >= 1 ? i - 1 : -1, 0});
    }
  for (auto& x : items) x.cost = 2LL * (x.i0 + 1) + 1 + (x.h1 >= 0 ? 2LL * (x.i1 + 1) + 1 : 0);
  std::stable_sort(items.begin(), items.end(), [](const PairItem& p, const PairItem& q) {
    if (p.cost != q.cost) return p.cost > q.cost;
    if (p.i0 != q.i0) return p.i0 > q.i0;
    if (p.b != q.b) return p.b < q.b;
    return p.kvh < q.kvh;
  });
  const long long n = (long long)items.size();
  const int grid = (int)(n < nsm ? n : nsm);
  std::vector<std::vector<int>> lists(grid);
  using Load = std::pair<long long, int>;  // (work so far, CTA): ties go to the lower CTA
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < grid; c++) heap.push(Load(0, c));
  for (long long w = 0; w < n; w++) {
    const Load l = heap.top();
    heap.pop();
    lists[l.second].push_back((int)w);
    heap.push(Load(l.first + items[w].cost, l.second));
  }
  int k = 0;
  for (auto& v : lists) k = (int)v.size() > k ? (int)v.size() : k;
  std::vector<int> table((size_t)grid * k * 4, -1);
  for (int c = 0; c < grid; c++)
    for (size_t j = 0; j < lists[c].size(); j++) {
      const PairItem& x = items[lists[c][j]];
      int* e = &table[((size_t)c * k + j) * 4];
      e[0] = x.b;
      e[1] = x.h0 | ((x.h1 + 1) << 16);
      e[2] = x.i0;
      e[3] = x.h1 >= 0 ? x.i1 : 0;
    }
  *grid_out = grid;
  *K = k;
  return table;
}

// Requires g_mu held.  The table is uploaded with a synchronous copy: make one
// call per shape before capturing calls in a graph.
int fwd_schedule(DeviceState& d, int B, int Hkv, int G, int nt, int nsm, const int** out, int* grid, int* K) {
  for (auto& x : d.scheds)
    if (x.B == B && x.Hkv == Hkv && x.G == G && x.nt == nt && x.nsm == nsm) {
      *out = x.ptr;
      *grid = x.grid;
      *K = x.K;
      return NE_OK;
    }
  int k = 0, gr = 0;
  const std::vector<int> table = fwd_pair_schedule(B, Hkv, G, nt, nsm, &gr, &k);
  int* p = nullptr;
  if (cudaMalloc(&p, sizeof(int) * table.size()) != cudaSuccess) return NE_ERR_CUDA;
  if (cudaMemcpy(p, table.data(), sizeof(int) * table.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(p);
    return NE_ERR_CUDA;
  }
  d.scheds.push_back(FwdSchedule{B, Hkv, G, nt, nsm, gr, k, p});
  *out = p;
  *grid = gr;
  *K = k;
  return NE_OK;
}

// Forward workspace owned by the library, one per stream, grown on demand.
// Never allocates while `s` is being captured into a graph (that would end the
// capture): a capture needs a workspace that is already large enough.
// Requires g_mu held.
int fwd_scratch(DeviceState& d, cudaStream_t s, size_t need, void** out) {
  FwdScratch* f = nullptr;
  for (auto& x : d.fwd_scratch)
    if (x.stream == s) f = &x;
  if (f && f->bytes >= need) {
    *out = f->ptr;
    return NE_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return NE_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return NE_ERR_WORKSPACE;
  if (!f) {
    d.fwd_scratch.push_back(FwdScratch{s, nullptr, 0});
    f = &d.fwd_scratch.back();
  }
  if (f->ptr) {
    // cudaFree waits for the device to finish the work that may still read it
    if (cudaFree(f->ptr) != cudaSuccess) return NE_ERR_CUDA;
    f->ptr = nullptr;
    f->bytes = 0;
  }
  if (cudaMalloc(&f->ptr, need) != cudaSuccess) {
    f->ptr = nullptr;
    return NE_ERR_CUDA;
  }
  f->bytes = need;
  *out = f->ptr;
  return NE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 4-D map over a [B, T, H, D] bf16 tensor; box = one head, 128 rows, all D.
int make_map_bthd(CUtensorMap* m, const void* ptr, int B, int T, int H, int D,
                  CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
  cuuint32_t box[4] = {(cuuint32_t)D, 1, (cuuint32_t)kTile, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, dt, 4, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        D == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 4-D map over a [B, T, H, D] e4m3 tensor (one byte per value); box = one head,
// 128 rows, all D (64 bytes per row for D = 64, 64-byte swizzle).
int make_map_bthd8(CUtensorMap* m, const void* ptr, int B, int T, int H, int D) {
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D, (cuuint64_t)H * D, (cuuint64_t)T * H * D};
  cuuint32_t box[4] = {(cuuint32_t)D, 1, (cuuint32_t)kTile, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 4-D map over a head-major key/value cache [B, H, Tcap, D] of which positions
// 0..Tkv-1 are valid: rows at or past Tkv read as zeros.  Box = 128 rows of one
// head, all D (one contiguous stretch).
int make_map_cache(CUtensorMap* m, const void* ptr, int B, int Tkv, int Tcap, int H, int D, CUtensorMapDataType dt) {
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Tkv, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Tcap * D * 2, (cuuint64_t)H * Tcap * D * 2};
  cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)kTile, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, dt, 4, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        D == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 4-D store map over a gradient [B, T, H, D] (fp32 or bf16); box = 128 bytes of
// columns (64 bytes when a row is that short) x 1 head x box_rows rows x 1, with
// the swizzle of that span.
int make_map_grad(CUtensorMap* m, void* ptr, int B, int T, int H, int D, bool fp32, int box_rows = kTile) {
  const int es = fp32 ? 4 : 2;
  const int span = D * es < 128 ? D * es : 128;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es, (cuuint64_t)T * H * D * es};
  cuuint32_t box[4] = {(cuuint32_t)(span / es), 1, (cuuint32_t)box_rows, 1};
  cuuint32_t e1[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims,
                        strides, box, e1, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 2-D map over the fp32 dQ accumulator [rows, D]; box = 32 columns x 128 rows.
int make_map_acc(CUtensorMap* m, void* ptr, long long rows, int D) {
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)kTile};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 2-D map over a row-major bf16 matrix [rows, cols]; box = 64 columns (128
// bytes) x box_rows rows, 128-byte swizzle (the UMMA K-major operand layout).
int make_map_rows(CUtensorMap* m, const void* ptr, long long rows, int cols, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// 4-D store map over a row-major [rows, H, D] tensor of 2-byte values (as
// {D, H, rows, 1}); box = 32 values of one head x 128 rows, 64-byte swizzle.
int make_map_out_box(CUtensorMap* m, void* ptr, long long rows, int H, int D, CUtensorMapDataType dt) {
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, 1};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)rows * H * D * 2};
  cuuint32_t box[4] = {32, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, dt, 4, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

int check_shape(int B, int T, int Hq, int Hkv, int D) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return NE_ERR_ARG;
  if (D != 32 && D != 64) return NE_ERR_UNSUPPORTED;
  const long long Tp = ((long long)T + kTile - 1) / kTile * kTile;
  const long long maxH = Hq > Hkv ? Hq : Hkv;
  if ((long long)B * Tp * maxH * D >= (1LL << 31)) return NE_ERR_UNSUPPORTED;
  const long long ntiles = Tp / kTile;
  if (ntiles * B * Hq >= (1LL << 31) - 1) return NE_ERR_UNSUPPORTED;
  if (Hq > 32767) return NE_ERR_UNSUPPORTED;  // the forward's work table packs two heads in 32 bits
  return NE_OK;
}

int heads_per_cta(int G, int D) {
  for (int hc = fwd_max_heads(D, true); hc >= 1; hc--)
    if (G % hc == 0) return hc;
  return 1;
}

struct WsLayout {
  size_t qr, kr, qlo, klo, lse2, lse2_lo, delta, dqacc, total;
};

// Workspace layouts.  Both start with the rotated fp16 q [B,T,Hq,D] and k
// [B,T,Hkv,D]: the forward's workspace is that prefix alone.
size_t ws_up(size_t x) { return (x + 255) / 256 * 256; }
size_t fwd_ws_bytes(int B, int T, int Hq, int Hkv, int D) {
  return ws_up(2 * (size_t)B * T * Hq * D) + ws_up(2 * (size_t)B * T * Hkv * D);
}
// FP8 forward workspace: e4m3 rotated q [B,T,Hq,D] and k [B,T,Hkv,D], then the
// per-head maxima [Hq + Hkv] (fp32).
size_t fwd8_ws_bytes(int B, int T, int Hq, int Hkv, int D) {
  return ws_up((size_t)B * T * Hq * D) + ws_up((size_t)B * T * Hkv * D) + ws_up(4 * (size_t)(Hq + Hkv));
}
constexpr int kFwdFlags = kFlagOFp32 | kFlagPreciseQK | kFlagRopeHalf | kFlagQKRotated | kFlagFp8;
// The FP8 forward: default precision, q and k rotated by the library, D = 64,
// at most 256 heads in all (per-head maxima of its first pass).
int fp8_rules(int flags, int Hq, int Hkv, int D) {
  if (!(flags & kFlagFp8)) return NE_OK;
  if (flags & (kFlagPreciseQK | kFlagQKRotated)) return NE_ERR_ARG;
  if (D != 64 || Hq + Hkv > 256) return NE_ERR_UNSUPPORTED;
  return NE_OK;
}

// Decode workspace: packed rotated queries, then the splits' partial O and (max, sum).
struct DecodeWs {
  size_t qpk, part_o, part_ml, done, total;
};
int decode_copies(int R) { return R <= 32 ? 4 : (R <= 64 ? 2 : 1); }
DecodeWs decode_ws(int B, int Tq, int Tkv, int Hq, int Hkv, int D) {
  const size_t R = (size_t)(Hq / Hkv) * Tq, ntk = ((size_t)Tkv + kTile - 1) / kTile;
  const size_t F = (size_t)decode_copies((int)R);
  DecodeWs w;
  w.qpk = 0;
  w.part_o = ws_up((size_t)B * Hkv * kTile * D * 2);
  w.part_ml = w.part_o + ws_up((size_t)B * Hkv * ntk * F * R * D * 4);
  w.done = w.part_ml + ws_up((size_t)B * Hkv * ntk * F * R * 8);
  w.total = w.done + ws_up((size_t)B * Hkv * 4);
  return w;
}

int check_decode_shape(int B, int Tq, int Tkv, int Tcap, int Hq, int Hkv, int D) {
  if (Tq < 1 || Tkv < Tq || Tcap < Tkv) return NE_ERR_ARG;
  int st = check_shape(B, Tcap, Hq, Hkv, D);
  if (st != NE_OK) return st;
  if ((Hq / Hkv) * Tq > kTile) return NE_ERR_UNSUPPORTED;
  return NE_OK;
}


// RMSNorm + projection: the attention shape rules, C % 8 == 0 (16-byte rows),
// and every row-major index within 2^31 elements.
int check_qkv_shape(int B, int T, int C, int Hq, int Hkv, int D) {
  int st = check_shape(B, T, Hq, Hkv, D);
  if (st != NE_OK) return st;
  if (C < 8 || C % 8 != 0) return NE_ERR_ARG;
  const long long M = (long long)B * T, N = (long long)(Hq + 2 * Hkv) * D;
  if ((M + 127) * C >= (1LL << 31) || N * C >= (1LL << 31) || M * N >= (1LL << 31)) return NE_ERR_UNSUPPORTED;
  return NE_OK;
}
// Workspace: [rotated q | rotated k] (the forward's workspace, with
// NE_ATTN_QK_ROTATED) then the folded projection matrix [N, C] bf16.
size_t qkv_wf_offset(int B, int T, int Hq, int Hkv, int D, int flags) {
  return (flags & kFlagQKRotated) ? fwd_ws_bytes(B, T, Hq, Hkv, D) : 0;
}
size_t qkv_ws_bytes(int B, int T, int C, int Hq, int Hkv, int D, int flags) {
  return qkv_wf_offset(B, T, Hq, Hkv, D, flags) + ws_up((size_t)(Hq + 2 * Hkv) * D * C * 2);
}

WsLayout ws_layout(int B, int T, int Hq, int Hkv, int D, bool precise) {
  auto up = ws_up;
  const size_t Tp = (size_t)(T + kTile - 1) / kTile * kTile;
  WsLayout w;
  size_t off = 0;
  w.qr = off;
  off += up(2 * (size_t)B * T * Hq * D);
  w.kr = off;
  off += up(2 * (size_t)B * T * Hkv * D);
  w.qlo = w.klo = 0;
  if (precise) {
    w.qlo = off;
    off += up(2 * (size_t)B * T * Hq * D);
    w.klo = off;
    off += up(2 * (size_t)B * T * Hkv * D);
  }
  w.dqacc = off;
  off += up(sizeof(float) * (size_t)B * Hq * Tp * D);
  w.lse2 = off;
  off += up(sizeof(float) * (size_t)B * Hq * Tp);
  w.lse2_lo = 0;
  if (precise) {
    w.lse2_lo = off;
    off += up(sizeof(float) * (size_t)B * Hq * Tp);
  }
  w.delta = off;
  off += up(sizeof(float) * (size_t)B * Hq * Tp);
  w.total = off;
  return w;
}

constexpr int kKnownFlags = kFlagOFp32 | kFlagGradFp32 | kFlagPreciseQK | kFlagRopeHalf;
// the split-precision kernels rotate tiles in shared memory in the interleaved layout only
bool half_with_precise(int flags) { return (flags & kFlagRopeHalf) && (flags & kFlagPreciseQK); }
constexpr int kBwdFlags = kKnownFlags | kFlagQKRotated;

// ------------------------------------------------------------------ kernel timing
struct Profile {
  bool on = false;
  int capacity = 0;
  int used = 0;
  std::vector<cudaEvent_t> ev;  // 2 * capacity
  std::vector<int> kind;        // per timed launch
  long long launches[NE_ATTN_NUM_KERNEL_KINDS] = {};
};
std::mutex g_prof_mu;
Profile g_prof;

void prof_reset() {
  for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
  g_prof = Profile();
}

// Under stream capture an event must be recorded as an external event node to be
// timed when the graph runs; otherwise a plain record.
void prof_record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

// Records the start event of a launch of `kind`; returns the slot (or -1).
int prof_begin(int kind, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof.on) return -1;
  g_prof.launches[kind]++;
  if (g_prof.used >= g_prof.capacity) return -1;
  const int slot = g_prof.used++;
  g_prof.kind[slot] = kind;
  prof_record(g_prof.ev[2 * slot], s);
  return slot;
}
void prof_end(int slot, cudaStream_t s) {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof.on && slot < g_prof.used) prof_record(g_prof.ev[2 * slot + 1], s);
}

struct ProfScope {
  int slot;
  cudaStream_t s;
  ProfScope(int kind, cudaStream_t st) : slot(prof_begin(kind, st)), s(st) {}
  ~ProfScope() { prof_end(slot, s); }
};

// The backward's three launches (pre-pass, dK/dV sweep, dq epilogue) on a
// workspace `ws` laid out as `w` with the rotary table `rope`; shared by
// ne_attn_bwd (caller workspace) and ne_attn_bwd_noalloc (the fixed array).
// Requires g_mu held.
int bwd_launch(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
               void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D, int flags, uint8_t* ws,
               const WsLayout& w, const float2* rope, int* status, cudaStream_t s) {
  int st;
  const bool precise = (flags & kFlagPreciseQK) != 0;
  const int grad_fp32 = (flags & kFlagGradFp32) ? 1 : 0;
  const int nt = (T + kTile - 1) / kTile;
  const int Tp = nt * kTile;
  float* dqacc = reinterpret_cast<float*>(ws + w.dqacc);
  __half* qr = reinterpret_cast<__half*>(ws + w.qr);
  __half* kr = reinterpret_cast<__half*>(ws + w.kr);
  __half* qlo = precise ? reinterpret_cast<__half*>(ws + w.qlo) : nullptr;
  __half* klo = precise ? reinterpret_cast<__half*>(ws + w.klo) : nullptr;
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2);
  float* lse2_lo = precise ? reinterpret_cast<float*>(ws + w.lse2_lo) : nullptr;
  float* delta = reinterpret_cast<float*>(ws + w.delta);
  const double scale = 1.0 / std::sqrt((double)D);

  PrepArgs p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.o = o;
  p.o_fp32 = (flags & kFlagOFp32) ? 1 : 0;
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.lse_lo = precise ? lse + (size_t)B * Hq * T : nullptr;
  p.lse2_lo = lse2_lo;
  p.qr = qr;
  p.kr = kr;
  p.qlo = qlo;
  p.klo = klo;
  p.lse2 = lse2;
  p.delta = delta;
  p.dqacc = dqacc;
  p.rope = rope;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.Tp = Tp;
  p.rotate_qk = (flags & kFlagQKRotated) ? 0 : 1;
  p.negate = precise ? 0 : 1;
  p.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
  p.div_hq = make_fastdiv((uint32_t)Hq);
  p.div_hkv = make_fastdiv((uint32_t)Hkv);
  p.div_t = make_fastdiv((uint32_t)T);
  p.div_pad = make_fastdiv((uint32_t)(Tp > T ? Tp - T : 1));
  {
    ProfScope prof(NE_ATTN_KERNEL_BWD_PREP, s);
    if (launch_bwd_prep(p, s) != cudaSuccess) return NE_ERR_CUDA;
  }

  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  constexpr CUtensorMapDataType kF16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if ((st = make_map_bthd(&a.map_qr, qr, B, T, Hq, D, kF16)) != NE_OK) return st;
  if ((st = make_map_bthd(&a.map_kr, kr, B, T, Hkv, D, kF16)) != NE_OK) return st;
  if ((st = make_map_bthd(&a.map_v, v, B, T, Hkv, D)) != NE_OK) return st;
  if ((st = make_map_bthd(&a.map_do, dout, B, T, Hq, D)) != NE_OK) return st;
  if (precise) {
    if ((st = make_map_bthd(&a.map_qlo, qlo, B, T, Hq, D, kF16)) != NE_OK) return st;
    if ((st = make_map_bthd(&a.map_klo, klo, B, T, Hkv, D, kF16)) != NE_OK) return st;
  }
  if ((st = make_map_acc(&a.map_dqacc, dqacc, (long long)B * Hq * Tp, D)) != NE_OK) return st;
  if ((st = make_map_grad(&a.map_dk, dk, B, T, Hkv, D, grad_fp32 != 0)) != NE_OK) return st;
  if ((st = make_map_grad(&a.map_dv, dv, B, T, Hkv, D, grad_fp32 != 0)) != NE_OK) return st;
  a.lse2 = lse2;
  a.lse2_lo = lse2_lo;
  a.delta = delta;
  a.dk = dk;
  a.dv = dv;
  a.rope = rope;
  a.status = status;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.G = Hq / Hkv;
  a.nt = nt;
  a.Tp = Tp;
  a.grad_fp32 = grad_fp32;
  a.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
  a.scale_log2 = (float)(1.4426950408889634 * scale);
  a.scale_log2_lo = (float)(1.4426950408889634 * scale - (double)a.scale_log2);
  a.scale = (float)scale;
  {
    ProfScope prof(NE_ATTN_KERNEL_BWD_DKDV, s);
    if (launch_bwd_dkdv(a, precise, s) != cudaSuccess) return NE_ERR_CUDA;
  }

  DqArgs qa;
  qa.dqacc = dqacc;
  qa.dq = dq;
  qa.rope = rope;
  qa.B = B;
  qa.T = T;
  qa.Hq = Hq;
  qa.D = D;
  qa.Tp = Tp;
  qa.grad_fp32 = grad_fp32;
  qa.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
  qa.scale = (float)scale;
  qa.div_hq = make_fastdiv((uint32_t)Hq);
  qa.div_hg = make_fastdiv((uint32_t)(Hq + 3) / 4);
  qa.div_t = make_fastdiv((uint32_t)T);
  {
    ProfScope prof(NE_ATTN_KERNEL_BWD_DQ, s);
    if (launch_bwd_dq(qa, s) != cudaSuccess) return NE_ERR_CUDA;
  }
  return NE_OK;
}

}  // namespace
}  // namespace ne

using namespace ne;

extern "C" {

size_t ne_attn_fwd_workspace_size(int B, int T, int Hq, int Hkv, int D, int flags) {
  if (check_shape(B, T, Hq, Hkv, D) != NE_OK || (flags & ~kFwdFlags) != 0) return 0;
  if (half_with_precise(flags) || ((flags & kFlagQKRotated) && (flags & kFlagPreciseQK))) return 0;
  if (fp8_rules(flags, Hq, Hkv, D) != NE_OK) return 0;
  if (flags & kFlagFp8) return fwd8_ws_bytes(B, T, Hq, Hkv, D);
  return (flags & kFlagPreciseQK) ? 0 : fwd_ws_bytes(B, T, Hq, Hkv, D);
}

int ne_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int Hq,
                   int Hkv, int D, float rope_base, int flags, void* workspace, size_t workspace_bytes,
                   void* stream) {
  const bool rotated = (flags & kFlagQKRotated) != 0;  // the workspace already holds the rotated q, k
  if ((!rotated && (!q || !k)) || !v || !o || !lse) return NE_ERR_ARG;
  if (!(rope_base > 1.0f) || !std::isfinite(rope_base)) return NE_ERR_ARG;
  if ((flags & ~kFwdFlags) != 0) return NE_ERR_ARG;
  if (rotated && (flags & kFlagPreciseQK)) return NE_ERR_ARG;
  if (half_with_precise(flags)) return NE_ERR_UNSUPPORTED;
  int st = check_shape(B, T, Hq, Hkv, D);
  if (st != NE_OK) return st;
  if ((st = fp8_rules(flags, Hq, Hkv, D)) != NE_OK) return st;
  const bool fp8 = (flags & kFlagFp8) != 0;
  if ((q && !aligned16(q)) || (k && !aligned16(k)) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return NE_ERR_ALIGN;
  const bool precise = (flags & kFlagPreciseQK) != 0;
  const size_t ws_need = precise ? 0 : (fp8 ? fwd8_ws_bytes(B, T, Hq, Hkv, D) : fwd_ws_bytes(B, T, Hq, Hkv, D));
  if ((rotated && !workspace) ||
      (workspace && (workspace_bytes < ws_need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)))
    return NE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  if ((st = current_device(&dev)) != NE_OK) return st;
  DeviceState* d;
  if ((st = device_state(dev, &d)) != NE_OK) return st;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.nt = (T + kTile - 1) / kTile;
  if ((st = rope_table(*d, D, (double)rope_base, a.nt * kTile, s, &a.rope)) != NE_OK) return st;
  if (!precise) {
    int nsm = 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1) return NE_ERR_CUDA;
    if ((st = fwd_schedule(*d, B, Hkv, Hq / Hkv, a.nt, nsm, &a.sched, &a.grid, &a.sched_k)) != NE_OK) return st;
  }
  if (precise) {
    if ((st = make_map_bthd(&a.map_q, q, B, T, Hq, D)) != NE_OK) return st;
    if ((st = make_map_bthd(&a.map_k, k, B, T, Hkv, D)) != NE_OK) return st;
  } else if (fp8) {
    void* ws = workspace;
    if (!ws && (st = fwd_scratch(*d, s, ws_need, &ws)) != NE_OK) return st;
    unsigned char* wb = static_cast<unsigned char*>(ws);
    RopeArgs ra;
    std::memset(&ra, 0, sizeof(ra));
    ra.q = static_cast<const __nv_bfloat16*>(q);
    ra.k = static_cast<const __nv_bfloat16*>(k);
    ra.q8 = wb;
    ra.k8 = wb + ws_up((size_t)B * T * Hq * D);
    ra.amax = reinterpret_cast<float*>(wb + ws_up((size_t)B * T * Hq * D) + ws_up((size_t)B * T * Hkv * D));
    ra.rope = a.rope;
    ra.B = B;
    ra.T = T;
    ra.Hq = Hq;
    ra.Hkv = Hkv;
    ra.div_hq = make_fastdiv((uint32_t)Hq);
    ra.div_hkv = make_fastdiv((uint32_t)Hkv);
    ra.div_t = make_fastdiv((uint32_t)T);
    ra.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
    if ((st = make_map_bthd8(&a.map_q, ra.q8, B, T, Hq, D)) != NE_OK) return st;
    if ((st = make_map_bthd8(&a.map_k, ra.k8, B, T, Hkv, D)) != NE_OK) return st;
    a.qk_amax = ra.amax;
    ProfScope prof(NE_ATTN_KERNEL_FWD_ROPE, s);
    if (cudaMemsetAsync(ra.amax, 0, sizeof(float) * (size_t)(Hq + Hkv), s) != cudaSuccess) return NE_ERR_CUDA;
    if (launch_rope_amax(ra, s) != cudaSuccess || launch_rope_q8(ra, s) != cudaSuccess) return NE_ERR_CUDA;
  } else {
    void* ws = workspace;
    if (!ws && (st = fwd_scratch(*d, s, ws_need, &ws)) != NE_OK) return st;
    RopeArgs ra;
    ra.q = static_cast<const __nv_bfloat16*>(q);
    ra.k = static_cast<const __nv_bfloat16*>(k);
    ra.qr = static_cast<__half*>(ws);
    ra.kr = reinterpret_cast<__half*>(static_cast<unsigned char*>(ws) + ws_up(2 * (size_t)B * T * Hq * D));
    ra.rope = a.rope;
    ra.B = B;
    ra.T = T;
    ra.Hq = Hq;
    ra.Hkv = Hkv;
    ra.div_hq = make_fastdiv((uint32_t)Hq);
    ra.div_hg = make_fastdiv((uint32_t)(Hq + Hkv + 3) / 4);
    ra.div_hkv = make_fastdiv((uint32_t)Hkv);
    ra.div_t = make_fastdiv((uint32_t)T);
    ra.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
    if ((st = make_map_bthd(&a.map_q, ra.qr, B, T, Hq, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != NE_OK) return st;
    if ((st = make_map_bthd(&a.map_k, ra.kr, B, T, Hkv, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != NE_OK) return st;
    if (!rotated) {
      ProfScope prof(NE_ATTN_KERNEL_FWD_ROPE, s);
      if (launch_rope_qk(ra, D, s) != cudaSuccess) return NE_ERR_CUDA;
    }
  }
  if ((st = make_map_bthd(&a.map_v, v, B, T, Hkv, D)) != NE_OK) return st;
  // the forward's warps store O 32 rows at a time
  if (!precise && (st = make_map_grad(&a.map_o, o, B, T, Hq, D, (flags & kFlagOFp32) != 0, 32)) != NE_OK) return st;
  a.o = o;
  a.lse = lse;
  a.status = d->status;
  a.B = B;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.G = Hq / Hkv;
  a.HC = precise ? heads_per_cta(a.G, D) : 1;
  a.o_fp32 = (flags & kFlagOFp32) ? 1 : 0;
  const double sl2 = 1.4426950408889634 / std::sqrt((double)D);
  a.scale_log2 = (float)sl2;
  a.scale_log2_lo = (float)(sl2 - (double)a.scale_log2);
  a.lse_lo = precise ? lse + (size_t)B * Hq * T : nullptr;
  ProfScope prof(NE_ATTN_KERNEL_FWD, s);
  return (fp8 ? launch_fwd_fp8(a, s) : launch_fwd(a, precise, s)) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

int ne_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int Hq, int Hkv,
                int D, float rope_base, void* stream) {
  return ne_attn_fwd_ex(q, k, v, o, lse, B, T, Hq, Hkv, D, rope_base, 0, nullptr, 0, stream);
}

size_t ne_attn_bwd_workspace_size(int B, int T, int Hq, int Hkv, int D, int flags) {
  if (check_shape(B, T, Hq, Hkv, D) != NE_OK || (flags & ~kBwdFlags) != 0) return 0;
  if ((flags & kFlagQKRotated) && (flags & kFlagPreciseQK)) return 0;
  if (half_with_precise(flags)) return 0;
  return ws_layout(B, T, Hq, Hkv, D, (flags & kFlagPreciseQK) != 0).total;
}

int ne_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D, float rope_base, int flags,
                void* workspace, size_t workspace_bytes, void* stream) {
  // with the rotated q, k in the workspace the kernels never read q and k
  const bool rotated = (flags & kFlagQKRotated) != 0;
  if ((!rotated && (!q || !k)) || !v || !o || !lse || !dout || !dq || !dk || !dv) return NE_ERR_ARG;
  if ((flags & ~kBwdFlags) != 0) return NE_ERR_ARG;
  // the forward leaves rotated copies only in default precision
  if (rotated && (flags & kFlagPreciseQK)) return NE_ERR_ARG;
  if (half_with_precise(flags)) return NE_ERR_UNSUPPORTED;
  if (!(rope_base > 1.0f) || !std::isfinite(rope_base)) return NE_ERR_ARG;
  int st = check_shape(B, T, Hq, Hkv, D);
  if (st != NE_OK) return st;
  if ((q && !aligned16(q)) || (k && !aligned16(k)) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return NE_ERR_ALIGN;
  const bool precise = (flags & kFlagPreciseQK) != 0;
  const WsLayout w = ws_layout(B, T, Hq, Hkv, D, precise);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return NE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  if ((st = current_device(&dev)) != NE_OK) return st;
  DeviceState* d;
  if ((st = device_state(dev, &d)) != NE_OK) return st;
  const int nt = (T + kTile - 1) / kTile;
  const int Tp = nt * kTile;
  const float2* rope = nullptr;
  if ((st = rope_table(*d, D, (double)rope_base, Tp, s, &rope)) != NE_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return bwd_launch(q, k, v, o, lse, dout, dq, dk, dv, B, T, Hq, Hkv, D, flags, ws, w, rope, d->status, s);
}

size_t ne_attn_qkv_workspace_size(int B, int T, int C, int Hq, int Hkv, int D, int flags) {
  if (check_qkv_shape(B, T, C, Hq, Hkv, D) != NE_OK || (flags & ~(kFlagQKRotated | kFlagRopeHalf)) != 0) return 0;
  return qkv_ws_bytes(B, T, C, Hq, Hkv, D, flags);
}

int ne_attn_qkv_rmsnorm(const void* x, const void* norm_w, const void* w_qkv, void* q, void* k, void* v,
                        float* rstd, int B, int T, int C, int Hq, int Hkv, int D, float eps, float rope_base,
                        int flags, void* workspace, size_t workspace_bytes, void* stream) {
  const bool rotated = (flags & kFlagQKRotated) != 0;
  if (!x || !norm_w || !w_qkv || !v || !rstd || (!rotated && (!q || !k))) return NE_ERR_ARG;
  if ((flags & ~(kFlagQKRotated | kFlagRopeHalf)) != 0) return NE_ERR_ARG;
  if (!(eps > 0.0f) || !std::isfinite(eps)) return NE_ERR_ARG;
  if (!(rope_base > 1.0f) || !std::isfinite(rope_base)) return NE_ERR_ARG;
  int st = check_qkv_shape(B, T, C, Hq, Hkv, D);
  if (st != NE_OK) return st;
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(w_qkv) || !aligned16(v) || !aligned16(rstd) ||
      (q && !aligned16(q)) || (k && !aligned16(k)))
    return NE_ERR_ALIGN;
  const size_t ws_need = qkv_ws_bytes(B, T, C, Hq, Hkv, D, flags);
  if ((rotated && !workspace) ||
      (workspace && (workspace_bytes < ws_need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)))
    return NE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev, nsm = 0;
  if ((st = current_device(&dev)) != NE_OK) return st;
  DeviceState* d;
  if ((st = device_state(dev, &d)) != NE_OK) return st;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1) return NE_ERR_CUDA;
  void* ws = workspace;
  if (!ws && (st = fwd_scratch(*d, s, ws_need, &ws)) != NE_OK) return st;
  QkvArgs a;
  std::memset(&a, 0, sizeof(a));
  if (rotated && (st = rope_table(*d, D, (double)rope_base, T, s, &a.rope)) != NE_OK) return st;
  unsigned char* wsb = static_cast<unsigned char*>(ws);
  a.M = B * T;
  a.C = C;
  a.N = (Hq + 2 * Hkv) * D;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.eps = eps;
  a.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.norm_w = static_cast<const __nv_bfloat16*>(norm_w);
  a.w = static_cast<const __nv_bfloat16*>(w_qkv);
  a.wf = reinterpret_cast<__nv_bfloat16*>(wsb + qkv_wf_offset(B, T, Hq, Hkv, D, flags));
  a.rstd = rstd;
  a.q = static_cast<__nv_bfloat16*>(q);
  a.k = static_cast<__nv_bfloat16*>(k);
  a.v = static_cast<__nv_bfloat16*>(v);
  if (rotated) {
    a.qr = reinterpret_cast<__half*>(wsb);
    a.kr = reinterpret_cast<__half*>(wsb + ws_up(2 * (size_t)B * T * Hq * D));
  }
  a.status = d->status;
  int grid = 1;
  const int BN = qkv_pick_bn(a.M, a.N, nsm, &grid);
  a.nkb = (C + 63) / 64;
  a.ntn = (a.N + BN - 1) / BN;
  a.tiles = ((a.M + 127) / 128) * a.ntn;
  if ((st = make_map_rows(&a.map_x, x, a.M, C, 128)) != NE_OK) return st;
  if ((st = make_map_rows(&a.map_w, a.wf, a.N, C, BN)) != NE_OK) return st;
  if ((st = make_map_out_box(&a.map_vst, v, a.M, Hkv, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)) != NE_OK) return st;
  if (rotated) {
    if ((st = make_map_out_box(&a.map_qr, a.qr, a.M, Hq, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != NE_OK) return st;
    if ((st = make_map_out_box(&a.map_kr, a.kr, a.M, Hkv, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != NE_OK) return st;
  }
  {
    ProfScope prof(NE_ATTN_KERNEL_QKV_PREP, s);
    if (launch_qkv_prep(a, s) != cudaSuccess) return NE_ERR_CUDA;
  }
  ProfScope prof(NE_ATTN_KERNEL_QKV, s);
  return launch_qkv_gemm(a, BN, grid, s) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

int ne_attn_check_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NE_ERR_CUDA;
  int dev;
  if (cudaGetDevice(&dev) != cudaSuccess) return NE_ERR_CUDA;
  DeviceState* d;
  int st;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if ((st = device_state(dev, &d)) != NE_OK) return st;
  }
  int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int)) != cudaSuccess) return NE_ERR_CUDA;
  if (word != 0 && cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return NE_ERR_CUDA;
  return word == 0 ? NE_OK : word;
}

const char* ne_attn_status_string(int status) {
  switch (status) {
    case NE_OK: return "ok";
    case NE_ERR_ARG: return "invalid argument (null pointer, bad size, Hq % Hkv != 0, rope_base or flags)";
    case NE_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case NE_ERR_UNSUPPORTED: return "unsupported (D not in {32, 64}, size limit, or device is not sm_103)";
    case NE_ERR_CUDA: return "CUDA runtime or launch error";
    case NE_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case NE_ERR_DEVICE_TIMEOUT: return "a kernel pipeline wait timed out on the device";
    case NE_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the fixed NE_ATTN_STATIC_SCRATCH_BYTES array of "
             "ne_attn_bwd_noalloc holds; use ne_attn_bwd with a caller workspace";
    default: return "unknown status";
  }
}

int ne_attn_profile_start(int capacity) {
  if (capacity < 0 || capacity > (1 << 22)) return NE_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  prof_reset();
  g_prof.ev.resize(2 * (size_t)capacity);
  g_prof.kind.resize(capacity);
  for (size_t i = 0; i < g_prof.ev.size(); i++) {
    if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
      g_prof.ev.resize(i);
      prof_reset();
      return NE_ERR_CUDA;
    }
  }
  g_prof.capacity = capacity;
  g_prof.on = true;
  return NE_OK;
}

int ne_attn_profile_stop(double* total_ms, long long* launches) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof.on) return NE_ERR_ARG;
  int st = NE_OK;
  double tot[NE_ATTN_NUM_KERNEL_KINDS] = {};
  for (int i = 0; i < g_prof.used; i++) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) {
      st = NE_ERR_CUDA;
      continue;
    }
    tot[g_prof.kind[i]] += ms;
  }
  for (int k = 0; k < NE_ATTN_NUM_KERNEL_KINDS; k++) {
    if (total_ms) total_ms[k] = tot[k];
    if (launches) launches[k] = g_prof.launches[k];
  }
  prof_reset();
  return st;
}

int ne_attn_profile_detach(void) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof.on) return NE_ERR_ARG;
  g_prof.on = false;  // no further launches are timed; the recorded events stay valid
  return NE_OK;
}

int ne_attn_profile_read(double* total_ms, long long* launches) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof.ev.empty()) return NE_ERR_ARG;
  int st = NE_OK;
  double tot[NE_ATTN_NUM_KERNEL_KINDS] = {};
  long long cnt[NE_ATTN_NUM_KERNEL_KINDS] = {};
  for (int i = 0; i < g_prof.used; i++) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) {
      st = NE_ERR_CUDA;
      continue;
    }
    tot[g_prof.kind[i]] += ms;
    cnt[g_prof.kind[i]]++;
  }
  for (int k = 0; k < NE_ATTN_NUM_KERNEL_KINDS; k++) {
    if (total_ms) total_ms[k] = tot[k];
    if (launches) launches[k] = cnt[k];
  }
  return st;
}

int ne_attn_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int B, int Tn,
                      int pos0, int Tcap, int Hkv, int D, float rope_base, int flags, void* stream) {
  if (!k_new || !v_new || !k_cache || !v_cache) return NE_ERR_ARG;
  if ((flags & ~kFlagRopeHalf) != 0) return NE_ERR_ARG;
  if (!(rope_base > 1.0f) || !std::isfinite(rope_base)) return NE_ERR_ARG;
  if (Tn < 1 || pos0 < 0 || (long long)pos0 + Tn > (long long)Tcap) return NE_ERR_ARG;
  int st = check_shape(B, Tcap, Hkv, Hkv, D);
  if (st != NE_OK) return st;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache)) return NE_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  if ((st = current_device(&dev)) != NE_OK) return st;
  DeviceState* d;
  if ((st = device_state(dev, &d)) != NE_OK) return st;
  KvAppendArgs a;
  std::memset(&a, 0, sizeof(a));
  if ((st = rope_table(*d, D, (double)rope_base, pos0 + Tn, s, &a.rope)) != NE_OK) return st;
  a.k = static_cast<const __nv_bfloat16*>(k_new);
  a.v = static_cast<const __nv_bfloat16*>(v_new);
  a.kc = static_cast<__half*>(k_cache);
  a.vc = static_cast<__nv_bfloat16*>(v_cache);
  a.B = B;
  a.Tn = Tn;
  a.Hkv = Hkv;
  a.Tcap = Tcap;
  a.pos0 = pos0;
  a.div_hkv = make_fastdiv((uint32_t)Hkv);
  a.div_tn = make_fastdiv((uint32_t)Tn);
  a.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
  ProfScope prof(NE_ATTN_KERNEL_KV_APPEND, s);
  return launch_kv_append(a, D, s) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

size_t ne_attn_decode_workspace_size(int B, int Tq, int Tkv, int Hq, int Hkv, int D) {
  if (check_decode_shape(B, Tq, Tkv, Tkv, Hq, Hkv, D) != NE_OK) return 0;
  return decode_ws(B, Tq, Tkv, Hq, Hkv, D).total;
}

int ne_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B, int Tq,
                   int Tkv, int Tcap, int Hq, int Hkv, int D, float rope_base, int flags, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !o || !lse) return NE_ERR_ARG;
  if (!(rope_base > 1.0f) || !std::isfinite(rope_base)) return NE_ERR_ARG;
  if ((flags & ~(kFlagOFp32 | kFlagRopeHalf)) != 0) return NE_ERR_ARG;
  int st = check_decode_shape(B, Tq, Tkv, Tcap, Hq, Hkv, D);
  if (st != NE_OK) return st;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse))
    return NE_ERR_ALIGN;
  const DecodeWs w = decode_ws(B, Tq, Tkv, Hq, Hkv, D);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return NE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev, nsm = 0;
  if ((st = current_device(&dev)) != NE_OK) return st;
  DeviceState* d;
  if ((st = device_state(dev, &d)) != NE_OK) return st;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1) return NE_ERR_CUDA;
  DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  if ((st = rope_table(*d, D, (double)rope_base, Tkv, s, &a.rope)) != NE_OK) return st;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.qpk = reinterpret_cast<__half*>(ws + w.qpk);
  a.part_o = reinterpret_cast<float*>(ws + w.part_o);
  a.part_ml = reinterpret_cast<float*>(ws + w.part_ml);
  a.done = reinterpret_cast<unsigned*>(ws + w.done);
  a.o = o;
  a.lse = lse;
  a.status = d->status;
  a.B = B;
  a.Tq = Tq;
  a.Tkv = Tkv;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.G = Hq / Hkv;
  a.R = a.G * Tq;
  a.F = decode_copies(a.R);
  a.rope_half = (flags & kFlagRopeHalf) ? 1 : 0;
  a.ntk = (Tkv + kTile - 1) / kTile;
  a.o_fp32 = (flags & kFlagOFp32) ? 1 : 0;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  // Splits of each (batch, key/value head)'s key tiles: the count whose slowest
  // CTA (work items per CTA x tiles per item, plus about one tile of fixed cost
  // per item) is shortest; among equals the smaller count, which leaves fewer
  // partial results to merge.
  const long long bh = (long long)B * Hkv;
  long long best = -1;
  for (int ns = 1; ns <= a.ntk && ns <= 64; ns++) {
    const long long cost = ((bh * ns + nsm - 1) / nsm) * ((a.ntk + ns - 1) / ns + 1);
    if (best < 0 || cost < best) {
      best = cost;
      a.nsplit = ns;
    }
  }
  if ((st = make_map_bthd(&a.map_q, a.qpk, 1, (int)(bh * kTile), 1, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != NE_OK)
    return st;
  if ((st = make_map_cache(&a.map_k, k_cache, B, Tkv, Tcap, Hkv, D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) != NE_OK)
    return st;
  if ((st = make_map_cache(&a.map_v, v_cache, B, Tkv, Tcap, Hkv, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)) != NE_OK)
    return st;
  {
    ProfScope prof(NE_ATTN_KERNEL_DECODE_AUX, s);
    if (launch_decode_q(a, s) != cudaSuccess) return NE_ERR_CUDA;
  }
  ProfScope prof(NE_ATTN_KERNEL_DECODE, s);
  return launch_decode(a, nsm, s) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

int ne_attn_debug_fwd_schedule(int B, int Hkv, int G, int nt, int nsm, int* table, int capacity, int* grid,
                               int* K) {
  if (B < 1 || Hkv < 1 || G < 1 || nt < 1 || nsm < 1 || !K || !grid) return NE_ERR_ARG;
  if ((long long)B * Hkv * G * nt >= (1LL << 31) || (long long)Hkv * G > 32767) return NE_ERR_ARG;
  const std::vector<int> t = fwd_pair_schedule(B, Hkv, G, nt, nsm, grid, K);
  if (!table || capacity < (long long)t.size()) return NE_ERR_ARG;
  std::memcpy(table, t.data(), sizeof(int) * t.size());
  return NE_OK;
}

int ne_attn_debug_timeout_probe(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return NE_ERR_ARG;
  int dev, st;
  if ((st = current_device(&dev)) != NE_OK) return st;
  DeviceState* d;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if ((st = device_state(dev, &d)) != NE_OK) return st;
  }
  return launch_timeout_probe(d->status, (long long)limit_us * 1000, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? NE_OK
             : NE_ERR_CUDA;
}

// Backward pass that allocates nothing: the same kernels as ne_attn_bwd, with
// their workspace and rotary table taken from the library's fixed device array
// instead of caller or library allocations.  See include/ne_attn.h.
int ne_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D,
                        float rope_base, int flags, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return NE_ERR_ARG;
  if ((flags & ~kKnownFlags) != 0) return NE_ERR_ARG;
  if (half_with_precise(flags)) return NE_ERR_UNSUPPORTED;
  if (!(rope_base > 1.0f) || !std::isfinite(rope_base)) return NE_ERR_ARG;
  int st = check_shape(B, T, Hq, Hkv, D);
  if (st != NE_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return NE_ERR_ALIGN;
  const bool precise = (flags & kFlagPreciseQK) != 0;
  const int nt = (T + kTile - 1) / kTile;
  const int Tp = nt * kTile;
  // scratch layout: [rotary table, Tp x D/2 float2][workspace as in ne_attn_bwd]
  const size_t table_bytes = (sizeof(float2) * (size_t)Tp * (D / 2) + 255) / 256 * 256;
  const WsLayout w = ws_layout(B, T, Hq, Hkv, D, precise);
  if (table_bytes + w.total > (size_t)NE_ATTN_STATIC_SCRATCH_BYTES) return NE_ERR_SCRATCH_LIMIT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev;
  if ((st = current_device(&dev)) != NE_OK) return st;
  DeviceState* d;
  if ((st = device_state(dev, &d)) != NE_OK) return st;
  if (!d->static_scratch) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return NE_ERR_CUDA;
    d->static_scratch = static_cast<unsigned char*>(p);
  }
  float2* rope = reinterpret_cast<float2*>(d->static_scratch);
  uint8_t* ws = d->static_scratch + table_bytes;
  // The array keeps the previous call's contents: the table is rebuilt here and
  // the pre-pass zeroes the dQ accumulator and writes every other field it uses.
  if (launch_rope_table(rope, Tp, D, (double)rope_base, s) != cudaSuccess) return NE_ERR_CUDA;
  return bwd_launch(q, k, v, o, lse, dout, dq, dk, dv, B, T, Hq, Hkv, D, flags, ws, w, rope, d->status, s);
}

}  // extern "C"
