// swasink.cu -- the C ABI of libswasink.so (see include/swasink.h): argument
// validation, kernel selection, tensor-map construction and launches.
//
// One translation unit holds every kernel so that the device error word is a
// single symbol without relocatable device code.
#include <cuda.h>
#include <cuda_runtime.h>

#include <array>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/swasink.h"
#include "decode.cuh"
#include "decode_tc.cuh"
#include "device_common.cuh"
#include "rope.cuh"
#include "simt_fwd.cuh"
#include "tc_global.cuh"
#include "tc_swa.cuh"
#include "topk.cuh"
#include "verify.cuh"
#include "verify_tc.cuh"

namespace {

thread_local char g_last_error[256] = "";
// CTA of the next sliding-window tensor-core launch from this thread whose
// loads are withheld (swa_test_withhold_loads); -1: none.
thread_local int g_withhold_cta = -1;

void set_cuda_error(const char* where, cudaError_t e) {
  snprintf(g_last_error, sizeof g_last_error, "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
}

void set_error_text(const char* text) { snprintf(g_last_error, sizeof g_last_error, "%s", text); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- per-device facts, looked up once ------------------------------------
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  bool tc_attr[2][2][2] = {};   // [bf16 output][4 heads per tile][D = 64]
  bool tcg_attr[2][2][2][4] = {};   // [bf16 output][scores][D = 64][heads per tile 1, 2, 4, 8]
  bool topk_attr = false;
  bool dectc_attr[5][2] = {};   // [log2 G][D = 64]
  bool vertc_attr[4][2][2] = {};   // [heads per group 1, 2, 4, 8][64 query rows][D = 64]
  bool decode_attr[2][2][5] = {};
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) {
    set_cuda_error("cudaGetDevice", e);
    return false;
  }
  if (*dev < 0 || *dev >= kMaxDevices) {
    set_error_text("device index out of range");
    return false;
  }
  return true;
}

bool device_sms(int dev, int* sms) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev[dev].ready) {
    int n = 0;
    cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      set_cuda_error("cudaDeviceGetAttribute", e);
      return false;
    }
    g_dev[dev].sms = n;
    g_dev[dev].ready = true;
  }
  *sms = g_dev[dev].sms;
  return true;
}

// ---- cuTensorMapEncodeTiled through the runtime's driver entry point ------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D row-major tensor [d3][d2][d1][d0] (d0 innermost), 128-byte swizzle.
bool make_map_4d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                 uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3, uint32_t b0, uint32_t b1,
                 uint32_t b2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error_text("cuTensorMapEncodeTiled unavailable");
    return false;
  }
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * esize, d0 * d1 * esize, d0 * d1 * d2 * esize};
  const cuuint32_t box[4] = {b0, b1, b2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return false;
  }
  return true;
}

swa_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_cuda_error(what, e);
    return SWA_ECUDA;
  }
  return SWA_OK;
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the kernel before it on the stream is finishing, and orders its
// memory accesses after that kernel itself (griddepcontrol.wait).
template <typename... KArgs, typename... Args>
swa_status launch_dependent(const char* what, void (*kern)(KArgs...), unsigned grid,
                            unsigned block, int smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e != cudaSuccess) {
    set_cuda_error(what, e);
    return SWA_ECUDA;
  }
  return check_launch(what);
}

enum FwdPath { kPathInvalid, kPathSimt, kPathTcSwa, kPathTcGlobal };

constexpr int kVerifyMaxL = 64;  // drafted tokens per verify call

bool verify_tc_applies(int L, int Hq, int Hkv, int D, int W, swa_dtype dt) {
  if (!(dt == SWA_BF16 && (D == 128 || D == 64) && W == swa::vertc::kW && Hkv >= 1 &&
        Hq % Hkv == 0 && L >= 1 && L <= swa::vertc::kLmax))
    return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G % swa::vertc::kG == 0;
}

// Query heads per sliding-window tile: 4 when G = 4, else 8 (a kv head's G =
// 8 R query heads then form R tile groups of 8 that share its keys).
int tc_heads_per_tile(int G) { return G == 4 ? 4 : 8; }

FwdPath select_fwd(int B, int T, int Hq, int Hkv, int D, int W, swa_dtype dt) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || Hq % Hkv) return kPathInvalid;
  if (dt != SWA_F32 && dt != SWA_BF16) return kPathInvalid;
  if (D != 64 && D != 128) return kPathInvalid;
  const int G = Hq / Hkv;
  if (dt == SWA_BF16) {
    // G = 8 R: R sets of CTAs walk the sibling groups in step (R <= 64)
    if (W <= swa::tcswa::kMaxW && (G == 4 || (G % swa::tcswa::kGroup == 0 && G <= 512)))
      return kPathTcSwa;   // D = 64 or 128
    // the online-softmax kernel takes any window: wider ones, and the group
    // sizes the sliding-window kernel's tiles do not fit (1, 2, above 512)
    if (G == 1 || G == 2 || G == 4 || G % swa::tcglobal::kG == 0)
      return kPathTcGlobal;   // D = 64 or 128
  }
  return kPathSimt;
}

template <typename Tin>
swa_status launch_simt(const void* q, const void* k, const void* v, const float* sink, float* out,
                       float* lse, int B, int T, int Hq, int Hkv, int D, int W,
                       cudaStream_t st) {
  const long long rows = (long long)B * T * Hq;
  const int warps_per_block = 8;
  const long long blocks = (rows + warps_per_block - 1) / warps_per_block;
  if (blocks > 0x7fffffffLL) {
    set_error_text("problem too large for the general kernel");
    return SWA_EUNSUPPORTED;
  }
  const float scale = (float)(1.0 / std::sqrt((double)D));
  const Tin* qq = static_cast<const Tin*>(q);
  const Tin* kk = static_cast<const Tin*>(k);
  const Tin* vv = static_cast<const Tin*>(v);
  if (D == 64)
    swa::simt_fwd_kernel<Tin, 64><<<(unsigned)blocks, warps_per_block * 32, 0, st>>>(
        qq, kk, vv, sink, out, lse, B, T, Hq, Hkv, W, scale);
  else
    swa::simt_fwd_kernel<Tin, 128><<<(unsigned)blocks, warps_per_block * 32, 0, st>>>(
        qq, kk, vv, sink, out, lse, B, T, Hq, Hkv, W, scale);
  return check_launch("simt_fwd_kernel");
}

// Tiles n_first .. n_first + n_tiles - 1 (of 128 / heads-per-tile positions
// each) of every sequence; n_tiles < 0: to the end of the sequence.
swa_status launch_tc_swa(const void* q, const void* k, const void* v, const float* sink,
                         void* out, float* lse, int B, int T, int Hq, int Hkv, int D, int W,
                         bool bf16_out, cudaStream_t st, int n_first = 0, int n_tiles = -1) {
  using namespace swa::tcswa;
  int dev, sms;
  if (!current_device(&dev) || !device_sms(dev, &sms)) return SWA_ECUDA;
  const int gt = tc_heads_per_tile(Hq / Hkv);
  const bool four = gt == 4, d64 = D == 64;
  const int kNpos = 128 / gt;
  void (*const kernels[2][2][2])(CUtensorMap, CUtensorMap, CUtensorMap, Params) = {
      {{swa_fwd_tc_kernel<false, 8, 128>, swa_fwd_tc_kernel<false, 8, 64>},
       {swa_fwd_tc_kernel<false, 4, 128>, swa_fwd_tc_kernel<false, 4, 64>}},
      {{swa_fwd_tc_kernel<true, 8, 128>, swa_fwd_tc_kernel<true, 8, 64>},
       {swa_fwd_tc_kernel<true, 4, 128>, swa_fwd_tc_kernel<true, 4, 64>}}};
  auto kern = kernels[bf16_out][four][d64];
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].tc_attr[bf16_out][four][d64]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
      if (e != cudaSuccess) {
        set_cuda_error("cudaFuncSetAttribute(swa_fwd_tc_kernel)", e);
        return SWA_ECUDA;
      }
      g_dev[dev].tc_attr[bf16_out][four][d64] = true;
    }
  }
  const int Hg = Hq / gt;
  const long long ntiles_seq = n_tiles >= 0 ? n_tiles : (T + kNpos - 1) / kNpos - n_first;
  const long long total_tiles = (long long)B * Hg * ntiles_seq;
  if (total_tiles >= (1LL << 31)) {
    set_error_text("problem too large for the tensor-core kernel");
    return SWA_EUNSUPPORTED;
  }
  if (total_tiles <= 0) return SWA_OK;
  CUtensorMap mq, mk, mv;
  if (!make_map_4d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, D, Hq, T, B, 64, gt, kNpos) ||
      !make_map_4d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, D, Hkv, T, B, 64, 1, kBlk) ||
      !make_map_4d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v, D, Hkv, T, B, 64, 1, kBlk))
    return SWA_ECUDA;
  Params p;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.W = W;
  p.Hg = Hg;
  p.rep = Hg / Hkv;
  p.n_first = n_first;
  p.ntiles_seq = (int)ntiles_seq;
  p.total_tiles = (int)total_tiles;
  p.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.withhold_cta = g_withhold_cta;   // one launch only
  g_withhold_cta = -1;
  // rep equal sets of CTAs, one per sibling group (the kernel's tile ranges)
  const long long per_set = total_tiles / p.rep;
  const long long cps = per_set < sms / p.rep ? per_set : sms / p.rep;
  const long long grid = cps * p.rep;
  kern<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, p);
  return check_launch("swa_fwd_tc_kernel");
}

// blockmax: optional block-score output; blk_idx: optional block list (sparse
// mode, query blocks of qb_size positions, topk entries each).
swa_status launch_tc_global(const void* q, const void* k, const void* v, const float* sink,
                            void* out, float* lse, int B, int T, int Hq, int Hkv, int D, int W,
                            bool bf16_out, cudaStream_t st, float* blockmax = nullptr,
                            const int* blk_idx = nullptr, int qb_size = 0, int topk = 0) {
  using namespace swa::tcglobal;
  int dev, sms;
  if (!current_device(&dev) || !device_sms(dev, &sms)) return SWA_ECUDA;
  const bool scores = blockmax != nullptr;
  const bool d64 = D == 64;
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const Params);
  // [bf16 output][scores][D = 64]
  // [bf16 output][scores][D = 64]: 8 heads per tile
  static const Kern kTable[2][2][2] = {
      {{swa_fwd_tc_global_kernel<false, false, 128, 8>, swa_fwd_tc_global_kernel<false, false, 64, 8>},
       {swa_fwd_tc_global_kernel<false, true, 128, 8>, swa_fwd_tc_global_kernel<false, true, 64, 8>}},
      {{swa_fwd_tc_global_kernel<true, false, 128, 8>, swa_fwd_tc_global_kernel<true, false, 64, 8>},
       {swa_fwd_tc_global_kernel<true, true, 128, 8>, swa_fwd_tc_global_kernel<true, true, 64, 8>}}};
  // [heads per tile 1, 2, 4][bf16 output][D = 64]: G = 1, 2 or 4, no block scores
  static const Kern kTableSmall[3][2][2] = {
      {{swa_fwd_tc_global_kernel<false, false, 128, 1>, swa_fwd_tc_global_kernel<false, false, 64, 1>},
       {swa_fwd_tc_global_kernel<true, false, 128, 1>, swa_fwd_tc_global_kernel<true, false, 64, 1>}},
      {{swa_fwd_tc_global_kernel<false, false, 128, 2>, swa_fwd_tc_global_kernel<false, false, 64, 2>},
       {swa_fwd_tc_global_kernel<true, false, 128, 2>, swa_fwd_tc_global_kernel<true, false, 64, 2>}},
      {{swa_fwd_tc_global_kernel<false, false, 128, 4>, swa_fwd_tc_global_kernel<false, false, 64, 4>},
       {swa_fwd_tc_global_kernel<true, false, 128, 4>, swa_fwd_tc_global_kernel<true, false, 64, 4>}}};
  const int G = Hq / Hkv;
  const int gt = G < kG ? G : kG;   // heads per tile: 1, 2, 4 or 8
  const int gi = gt == 1 ? 0 : gt == 2 ? 1 : gt == 4 ? 2 : 3;
  if (gt != kG && (scores || blk_idx != nullptr)) {
    set_error_text("block scores and sparse mode take 8 heads per kv head");
    return SWA_EUNSUPPORTED;
  }
  const Kern kern = gt != kG ? kTableSmall[gi][bf16_out][d64] : kTable[bf16_out][scores][d64];
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].tcg_attr[bf16_out][scores][d64][gi]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
      if (e != cudaSuccess) {
        set_cuda_error("cudaFuncSetAttribute(swa_fwd_tc_global_kernel)", e);
        return SWA_ECUDA;
      }
      g_dev[dev].tcg_attr[bf16_out][scores][d64][gi] = true;
    }
  }
  const int item_pos = item_pos_for(gt), npos = npos_for(gt);
  const long long nitem_seq = (T + item_pos - 1) / item_pos;
  const int Hg = Hq / gt;   // head groups of a tile; the scores and sparse modes have Hg = Hkv
  const long long total = (long long)B * Hg * nitem_seq;
  if (total >= (1LL << 31)) {
    set_error_text("problem too large for the tensor-core kernel");
    return SWA_EUNSUPPORTED;
  }
  CUtensorMap mq, mk, mv;
  if (!make_map_4d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, D, Hq, T, B, 64, gt, npos) ||
      !make_map_4d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k, D, Hkv, T, B, 64, 1, kBlk) ||
      !make_map_4d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v, D, Hkv, T, B, 64, 1, kBlk))
    return SWA_ECUDA;
  Params p;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.W = W;
  p.Hg = Hg;
  p.rep = Hg / Hkv;
  p.item_pos = item_pos;
  p.nitem_seq = (int)nitem_seq;
  p.total_items = (int)total;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.blockmax = blockmax;
  p.nqg = (T + 3) / 4;
  p.nkb = (T + kBlk - 1) / kBlk;
  p.blk_idx = blk_idx;
  p.qb_size = qb_size > 0 ? qb_size : item_pos;
  p.topk = topk;
  p.nqb = (T + p.qb_size - 1) / p.qb_size;
  const long long grid = total < sms ? total : sms;
  kern<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, p);
  return check_launch("swa_fwd_tc_global_kernel");
}

template <typename Tin, int D, int G>
swa_status launch_decode_t(const void* q, const void* kr, const void* vr, const int64_t* pos,
                           const float* sink, float* out, float* lse, int B, int Hq, int Hkv,
                           int W, int rep, cudaStream_t st, bool* attr_done) {
  const swa::DecodeSmem L = swa::decode_smem_layout<Tin, D, G>(W);
  auto kern = swa::decode_kernel<Tin, D, G>;
  if (!*attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) {
      set_cuda_error("cudaFuncSetAttribute(decode_kernel)", e);
      return SWA_ECUDA;
    }
    *attr_done = true;
  }
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  kern<<<(unsigned)(B * Hkv * rep), swa::kDecodeThreads, L.total, st>>>(
      static_cast<const Tin*>(q), static_cast<const Tin*>(kr), static_cast<const Tin*>(vr), pos,
      sink, out, lse, Hq, Hkv, W, rep, scale_log2);
  return check_launch("decode_kernel");
}

// Tensor-core decode: bf16, D = 64 or 128, W = 128, G = 1, 2, 4, 8 or 16 query
// heads per kv head, or a larger multiple of 8 (R = G / 8 sibling groups of 8
// per kv head on the 8-head instance).  Returns log2 of the instance's heads
// per group and sets *rep = R (1 otherwise); -1 for other G.
int log2_group(int Hq, int Hkv, int* rep = nullptr) {
  if (rep) *rep = 1;
  if (Hkv < 1 || Hq % Hkv) return -1;
  const int G = Hq / Hkv;
  switch (G) {
    case 1: return 0;
    case 2: return 1;
    case 4: return 2;
    case 8: return 3;
    case 16: return 4;
    default:
      if (G % 8 != 0) return -1;
      if (rep) *rep = G / 8;
      return 3;
  }
}

bool decode_tc_applies(int Hq, int Hkv, int D, int W, swa_dtype dt) {
  return dt == SWA_BF16 && (D == 128 || D == 64) && W == swa::dectc::kW &&
         log2_group(Hq, Hkv) >= 0;
}

swa_status launch_decode_tc(const void* q, const void* kr, const void* vr, const int64_t* pos,
                            const float* sink, float* out, float* lse, int B, int Hq, int Hkv,
                            int D, cudaStream_t st, int dev) {
  using namespace swa::dectc;
  int sms;
  if (!device_sms(dev, &sms)) return SWA_ECUDA;
  int rep = 1;
  const int lg = log2_group(Hq, Hkv, &rep);
  const bool d64 = D == 64;
  void (*const kernels[5][2])(CUtensorMap, CUtensorMap, CUtensorMap, Params) = {
      {decode_tc_kernel<1, 128>, decode_tc_kernel<1, 64>},
      {decode_tc_kernel<2, 128>, decode_tc_kernel<2, 64>},
      {decode_tc_kernel<4, 128>, decode_tc_kernel<4, 64>},
      {decode_tc_kernel<8, 128>, decode_tc_kernel<8, 64>},
      {decode_tc_kernel<16, 128>, decode_tc_kernel<16, 64>}};
  if (lg < 0) return SWA_EUNSUPPORTED;
  auto kern = kernels[lg][d64];
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].dectc_attr[lg][d64]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemBytes);
      if (e != cudaSuccess) {
        set_cuda_error("cudaFuncSetAttribute(decode_tc_kernel)", e);
        return SWA_ECUDA;
      }
      g_dev[dev].dectc_attr[lg][d64] = true;
    }
  }
  const long long rings = (long long)B * Hkv;          // ring units (sequence, kv head)
  const long long units = rings * rep;                 // groups of the instance's heads
  if (rings * kW >= (1LL << 31) || units >= (1LL << 31) || (long long)B * Hq >= (1LL << 31)) {
    set_error_text("problem too large for the tensor-core decode kernel");
    return SWA_EUNSUPPORTED;
  }
  CUtensorMap mk, mv, mq;
  if (!make_map_4d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kr, D, rings * kW, 1, 1, 64, kW, 1) ||
      !make_map_4d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vr, D, rings * kW, 1, 1, 64, kW, 1) ||
      !make_map_4d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, D, (uint64_t)B * Hq, 1, 1, 64, kN,
                   1))
    return SWA_ECUDA;
  Params p;
  p.pos = pos;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.rep = rep;
  p.units = (int)units;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  const long long grid = units < sms ? units : sms;
  return launch_dependent("decode_tc_kernel", kern, (unsigned)grid, threads_for(1 << lg, D), kSmemBytes,
                          st, mk, mv, mq, p);
}

swa_status launch_verify_tc(const void* q, const void* kn, const void* vn, const void* kr,
                            const void* vr, const int64_t* pos, const float* sink, float* out,
                            float* lse, int B, int L, int Hq, int Hkv, int D, cudaStream_t st) {
  using namespace swa::vertc;
  int dev, sms;
  if (!current_device(&dev) || !device_sms(dev, &sms)) return SWA_ECUDA;
  // query heads per group: G = 1, 2, 4, else 8 (R sibling groups for G = 8 R);
  // 32 query rows per group up to 32 (8 heads: L <= 4), else 64
  const int G = Hq / Hkv;
  const int gv = G < kG ? G : kG;
  const int gi = gv == 1 ? 0 : gv == 2 ? 1 : gv == 4 ? 2 : 3;
  const bool rows64 = L * gv > 32, d64 = D == 64;
  using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, Params);
  // [heads per group 1, 2, 4, 8][64 query rows][D = 64]
  static const Kern kernels[4][2][2] = {
      {{verify_tc_kernel<32, 128, 1>, verify_tc_kernel<32, 64, 1>}, {nullptr, nullptr}},
      {{verify_tc_kernel<32, 128, 2>, verify_tc_kernel<32, 64, 2>}, {nullptr, nullptr}},
      {{verify_tc_kernel<32, 128, 4>, verify_tc_kernel<32, 64, 4>}, {nullptr, nullptr}},
      {{verify_tc_kernel<32, 128, 8>, verify_tc_kernel<32, 64, 8>},
       {verify_tc_kernel<64, 128, 8>, verify_tc_kernel<64, 64, 8>}}};
  const Kern kern = kernels[gi][rows64][d64];
  if (kern == nullptr) return SWA_EUNSUPPORTED;   // L * G <= 32 below 8 heads (L <= 8)
  const int smem = rows64 ? Layout<64>::kSmemBytes : Layout<32>::kSmemBytes;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].vertc_attr[gi][rows64][d64]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           smem);
      if (e != cudaSuccess) {
        set_cuda_error("cudaFuncSetAttribute(verify_tc_kernel)", e);
        return SWA_ECUDA;
      }
      g_dev[dev].vertc_attr[gi][rows64][d64] = true;
    }
  }
  const int rep = G / gv;                              // query groups per kv head
  const long long rings = (long long)B * Hkv;          // ring units (sequence, kv head)
  const long long units = rings * rep;
  if (rings * kW >= (1LL << 31) || units >= (1LL << 31)) {
    set_error_text("problem too large for the tensor-core verify kernel");
    return SWA_EUNSUPPORTED;
  }
  CUtensorMap mk, mv, mq, mkn, mvn;
  if (!make_map_4d(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kr, D, rings * kW, 1, 1, 64, kW, 1) ||
      !make_map_4d(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vr, D, rings * kW, 1, 1, 64, kW, 1) ||
      !make_map_4d(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, D, Hq, L, B, 64, gv, L) ||
      !make_map_4d(&mkn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kn, D, Hkv, L, B, 64, 1, L) ||
      !make_map_4d(&mvn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vn, D, Hkv, L, B, 64, 1, L))
    return SWA_ECUDA;
  Params p;
  p.pos = pos;
  p.sink = sink;
  p.out = out;
  p.lse = lse;
  p.B = B;
  p.L = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.rep = rep;
  p.units = (int)units;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  const long long grid = units < sms ? units : sms;
  return launch_dependent("verify_tc_kernel", kern, (unsigned)grid, kThreads, smem, st, mk, mv, mq, mkn, mvn, p);
}

template <typename Tin, int D>
swa_status launch_decode_g(const void* q, const void* kr, const void* vr, const int64_t* pos,
                           const float* sink, float* out, float* lse, int B, int Hq, int Hkv,
                           int W, cudaStream_t st, int dev) {
  // heads per CTA: the largest of 16, 8, 4, 2, 1 that divides G; a kv head's
  // G heads then run as rep = G / Gc sibling CTAs
  const int G = Hq / Hkv;
  const int Gc = G % 16 == 0 ? 16 : G % 8 == 0 ? 8 : G % 4 == 0 ? 4 : G % 2 == 0 ? 2 : 1;
  const int rep = G / Gc;
  if ((long long)B * Hkv * rep >= (1LL << 31)) {
    set_error_text("problem too large for the decode kernel");
    return SWA_EUNSUPPORTED;
  }
  const int ti = std::is_same<Tin, float>::value ? 0 : 1;
  const int di = D == 64 ? 0 : 1;
  bool* attr = nullptr;
  const int gi = Gc == 1 ? 0 : Gc == 2 ? 1 : Gc == 4 ? 2 : Gc == 8 ? 3 : 4;
  bool done;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    done = g_dev[dev].decode_attr[ti][di][gi];
  }
  attr = &done;
  swa_status s;
  switch (Gc) {
    case 1: s = launch_decode_t<Tin, D, 1>(q, kr, vr, pos, sink, out, lse, B, Hq, Hkv, W, rep, st, attr); break;
    case 2: s = launch_decode_t<Tin, D, 2>(q, kr, vr, pos, sink, out, lse, B, Hq, Hkv, W, rep, st, attr); break;
    case 4: s = launch_decode_t<Tin, D, 4>(q, kr, vr, pos, sink, out, lse, B, Hq, Hkv, W, rep, st, attr); break;
    case 8: s = launch_decode_t<Tin, D, 8>(q, kr, vr, pos, sink, out, lse, B, Hq, Hkv, W, rep, st, attr); break;
    default: s = launch_decode_t<Tin, D, 16>(q, kr, vr, pos, sink, out, lse, B, Hq, Hkv, W, rep, st, attr); break;
  }
  if (done) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    g_dev[dev].decode_attr[ti][di][gi] = true;
  }
  return s;
}

}  // namespace

extern "C" {

swa_status swa_sink_fwd_ex(const void* q, const void* k, const void* v, const float* sink,
                           void* out, float* lse, int B, int T, int Hq, int Hkv, int D, int W,
                           swa_dtype in_dtype, swa_dtype out_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!q || !k || !v || !sink || !out) return SWA_EINVAL;
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || Hq % Hkv) return SWA_EINVAL;
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return SWA_EINVAL;
  if (out_dtype != SWA_F32 && out_dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (lse && !aligned16(lse)))
    return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16_out = out_dtype == SWA_BF16;
  switch (select_fwd(B, T, Hq, Hkv, D, W, in_dtype)) {
    case kPathTcSwa:
      return launch_tc_swa(q, k, v, sink, out, lse, B, T, Hq, Hkv, D, W, bf16_out, st);
    case kPathTcGlobal:
      return launch_tc_global(q, k, v, sink, out, lse, B, T, Hq, Hkv, D, W, bf16_out, st);
    case kPathSimt:
      if (bf16_out) {
        set_error_text("bf16 output is available on the tensor-core paths only");
        return SWA_EUNSUPPORTED;
      }
      if (in_dtype == SWA_F32)
        return launch_simt<float>(q, k, v, sink, static_cast<float*>(out), lse, B, T, Hq, Hkv,
                                  D, W, st);
      return launch_simt<__nv_bfloat16>(q, k, v, sink, static_cast<float*>(out), lse, B, T, Hq,
                                        Hkv, D, W, st);
    default:
      return SWA_EINVAL;
  }
}

swa_status swa_sink_fwd(const void* q, const void* k, const void* v, const float* sink,
                        float* out, float* lse, int B, int T, int Hq, int Hkv, int D, int W,
                        swa_dtype in_dtype, void* stream) {
  return swa_sink_fwd_ex(q, k, v, sink, out, lse, B, T, Hq, Hkv, D, W, in_dtype, SWA_F32, stream);
}

// ---- prefill from and to host memory: per-chunk copy in / compute / copy out ----
namespace {
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> ev;   // [0] start, [1] end, then per chunk: in, computed
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

bool pipe_events(HostPipe& hp, size_t n) {
  while (hp.ev.size() < n) {
    cudaEvent_t e;
    cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (r != cudaSuccess) {
      set_cuda_error("cudaEventCreateWithFlags", r);
      return false;
    }
    hp.ev.push_back(e);
  }
  return true;
}

bool pipe_ready(HostPipe& hp) {
  if (hp.ready) return true;
  cudaError_t r = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
  if (r == cudaSuccess) r = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
  if (r != cudaSuccess) {
    set_cuda_error("cudaStreamCreateWithFlags", r);
    return false;
  }
  hp.ready = true;
  return true;
}

swa_status cuda_ok(cudaError_t r, const char* what) {
  if (r == cudaSuccess) return SWA_OK;
  set_cuda_error(what, r);
  return SWA_ECUDA;
}

char* byte_at(const void* base, size_t off) {
  return const_cast<char*>(static_cast<const char*>(base)) + off;
}

// The sliding-window tensor-core path: chunks of one sequence x a range of
// positions, staged in the device buffers at their own places, so that every
// copy is one contiguous range (the lse, [B, Hq, T], goes as Hq rows).  The
// prefill of a chunk computes its tiles only; the keys of the window before
// its first position came in with earlier chunks of the same sequence, on the
// same stream, so they are in place when it runs.
swa_status host_by_position(const void* q_h, const void* k_h, const void* v_h, const float* sink,
                            void* out_h, float* lse_h, void* q_d, void* k_d, void* v_d,
                            void* out_d, float* lse_d, int B, int T, int Hq, int Hkv, int D,
                            int W, bool bf16_out, cudaStream_t st, HostPipe& hp) {
  // chunks of whole tiles for either tile shape (16 or 32 positions)
  const int kNpos = 128 / tc_heads_per_tile(Hq / Hkv), kChunkAlign = 32;
  if (!aligned16(q_d) || !aligned16(k_d) || !aligned16(v_d) || !aligned16(out_d) ||
      (lse_d && !aligned16(lse_d)))
    return SWA_EINVAL;
  // about 16 chunks in all, of at least 512 positions, whole tiles except the last
  int nper = (16 + B - 1) / B;
  if (nper > T / 512) nper = T / 512;
  if (nper < 1) nper = 1;
  const int Tc = ((T + nper - 1) / nper + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
  // chunks {b, t0, t1}; the copy-in of the first and the copy-out of the last
  // overlap nothing, so a short piece (kEdge positions) is split off each
  constexpr int kEdge = 512;
  std::vector<std::array<int, 3>> chunks;
  for (int b = 0; b < B; ++b)
    for (int t0 = 0; t0 < T; t0 += Tc) chunks.push_back({b, t0, t0 + Tc < T ? t0 + Tc : T});
  if (chunks.front()[2] - chunks.front()[1] > 2 * kEdge) {
    const std::array<int, 3> f = chunks.front();
    chunks.front()[2] = f[1] + kEdge;
    chunks.insert(chunks.begin() + 1, {f[0], f[1] + kEdge, f[2]});
  }
  if (chunks.back()[2] - chunks.back()[1] > 2 * kEdge) {
    const std::array<int, 3> l = chunks.back();
    const int cut = (l[2] - kEdge) / kChunkAlign * kChunkAlign;   // a tile boundary
    chunks.back()[2] = cut;
    chunks.push_back({l[0], cut, l[2]});
  }
  const int nchunk = (int)chunks.size();
  const size_t q_tok = (size_t)Hq * D * 2, k_tok = (size_t)Hkv * D * 2;
  const size_t o_tok = (size_t)Hq * D * (bf16_out ? 2 : 4);
  if (!pipe_events(hp, 2 + 2 * (size_t)nchunk)) return SWA_ECUDA;
  cudaEvent_t ev_start = hp.ev[0], ev_end = hp.ev[1];
  swa_status rc = cuda_ok(cudaEventRecord(ev_start, st), "cudaEventRecord");
  if (rc == SWA_OK) rc = cuda_ok(cudaStreamWaitEvent(hp.h2d, ev_start, 0), "cudaStreamWaitEvent");
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  for (int c = 0; rc == SWA_OK && c < nchunk; ++c) {
    const int b = chunks[c][0], t0 = chunks[c][1], t1 = chunks[c][2];
    const size_t row0 = (size_t)b * T + t0, n = (size_t)(t1 - t0), seq0 = (size_t)b * T;
    cudaEvent_t ev_in = hp.ev[2 + 2 * c], ev_c = hp.ev[3 + 2 * c];
    rc = cuda_ok(cudaMemcpyAsync(byte_at(q_d, row0 * q_tok), byte_at(q_h, row0 * q_tok),
                                 n * q_tok, h2d, hp.h2d),
                 "cudaMemcpyAsync(q)");
    if (rc == SWA_OK)
      rc = cuda_ok(cudaMemcpyAsync(byte_at(k_d, row0 * k_tok), byte_at(k_h, row0 * k_tok),
                                   n * k_tok, h2d, hp.h2d),
                   "cudaMemcpyAsync(k)");
    if (rc == SWA_OK)
      rc = cuda_ok(cudaMemcpyAsync(byte_at(v_d, row0 * k_tok), byte_at(v_h, row0 * k_tok),
                                   n * k_tok, h2d, hp.h2d),
                   "cudaMemcpyAsync(v)");
    if (rc == SWA_OK) rc = cuda_ok(cudaEventRecord(ev_in, hp.h2d), "cudaEventRecord");
    if (rc == SWA_OK) rc = cuda_ok(cudaStreamWaitEvent(st, ev_in, 0), "cudaStreamWaitEvent");
    if (rc == SWA_OK)
      rc = launch_tc_swa(byte_at(q_d, seq0 * q_tok), byte_at(k_d, seq0 * k_tok),
                         byte_at(v_d, seq0 * k_tok), sink, byte_at(out_d, seq0 * o_tok),
                         lse_d ? lse_d + (size_t)b * Hq * T : nullptr, 1, T, Hq, Hkv, D, W,
                         bf16_out, st, t0 / kNpos, (t1 + kNpos - 1) / kNpos - t0 / kNpos);
    if (rc == SWA_OK) rc = cuda_ok(cudaEventRecord(ev_c, st), "cudaEventRecord");
    if (rc == SWA_OK) rc = cuda_ok(cudaStreamWaitEvent(hp.d2h, ev_c, 0), "cudaStreamWaitEvent");
    if (rc == SWA_OK)
      rc = cuda_ok(cudaMemcpyAsync(byte_at(out_h, row0 * o_tok), byte_at(out_d, row0 * o_tok),
                                   n * o_tok, d2h, hp.d2h),
                   "cudaMemcpyAsync(out)");
    if (rc == SWA_OK && lse_d)
      rc = cuda_ok(cudaMemcpy2DAsync(lse_h + (size_t)b * Hq * T + t0, (size_t)T * 4,
                                     lse_d + (size_t)b * Hq * T + t0, (size_t)T * 4, n * 4, Hq,
                                     d2h, hp.d2h),
                   "cudaMemcpy2DAsync(lse)");
  }
  // later work on `stream` follows every copy enqueued above, even after an error
  const swa_status rc_end = cuda_ok(cudaEventRecord(ev_end, hp.d2h), "cudaEventRecord");
  const swa_status rc_wait =
      rc_end == SWA_OK ? cuda_ok(cudaStreamWaitEvent(st, ev_end, 0), "cudaStreamWaitEvent")
                       : rc_end;
  return rc != SWA_OK ? rc : rc_wait;
}
}  // namespace

swa_status swa_sink_fwd_host(const void* q_h, const void* k_h, const void* v_h,
                             const float* sink, void* out_h, float* lse_h, void* q_d,
                             void* k_d, void* v_d, void* out_d, float* lse_d, int B, int T,
                             int Hq, int Hkv, int D, int W, swa_dtype in_dtype,
                             swa_dtype out_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!q_h || !k_h || !v_h || !out_h || !q_d || !k_d || !v_d || !out_d || !sink)
    return SWA_EINVAL;
  if ((lse_h == nullptr) != (lse_d == nullptr)) return SWA_EINVAL;
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || Hq % Hkv) return SWA_EINVAL;
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return SWA_EINVAL;
  if (out_dtype != SWA_F32 && out_dtype != SWA_BF16) return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  if (select_fwd(B, T, Hq, Hkv, D, W, in_dtype) == kPathTcSwa) {
    int dev;
    if (!current_device(&dev)) return SWA_ECUDA;
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe& hp = g_pipe[dev];
    if (!pipe_ready(hp)) return SWA_ECUDA;
    return host_by_position(q_h, k_h, v_h, sink, out_h, lse_h, q_d, k_d, v_d, out_d, lse_d, B, T,
                            Hq, Hkv, D, W, out_dtype == SWA_BF16,
                            static_cast<cudaStream_t>(stream), hp);
  }
  const size_t ie = in_dtype == SWA_BF16 ? 2 : 4, oe = out_dtype == SWA_BF16 ? 2 : 4;
  // Other paths: chunks of one sequence x a share of the kv heads (two shares when Hkv is
  // even), each staged compactly in the caller's device buffers.  Smaller
  // chunks shorten the copy-in before the first prefill and the copy-out after
  // the last, the two that overlap nothing.  When a share's staging offsets
  // would lose the 16-byte alignment the kernels need, the batch goes as one
  // chunk.
  int nsplit = (Hkv % 2 == 0) ? 2 : 1, nseq = 1;
  auto chunking_ok = [&](int ns, int nq) {
    const size_t hq = (size_t)Hq / ns, hk = (size_t)Hkv / ns;
    return ((size_t)nq * T * hq * D * ie) % 16 == 0 && ((size_t)nq * T * hk * D * ie) % 16 == 0 &&
           ((size_t)nq * T * hq * D * oe) % 16 == 0 &&
           (!lse_d || ((size_t)nq * hq * T * 4) % 16 == 0);
  };
  if (!chunking_ok(nsplit, 1)) nsplit = 1;
  if (!chunking_ok(nsplit, 1)) nseq = B;   // a single chunk: the whole batch
  const int Hq_c = Hq / nsplit, Hkv_c = Hkv / nsplit;
  const size_t q_row = (size_t)Hq_c * D * ie, k_row = (size_t)Hkv_c * D * ie;
  const size_t o_row = (size_t)Hq_c * D * oe;
  const size_t q_pitch = (size_t)Hq * D * ie, k_pitch = (size_t)Hkv * D * ie;
  const size_t o_pitch = (size_t)Hq * D * oe;
  const size_t q_chunk = (size_t)nseq * T * q_row, k_chunk = (size_t)nseq * T * k_row;
  const size_t o_chunk = (size_t)nseq * T * o_row, l_chunk = (size_t)nseq * Hq_c * T * 4;
  const int nchunk = (B / nseq) * nsplit;
  int dev;
  if (!current_device(&dev)) return SWA_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe& hp = g_pipe[dev];
  if (!pipe_ready(hp) || !pipe_events(hp, 2 + 2 * (size_t)nchunk)) return SWA_ECUDA;
  cudaEvent_t ev_start = hp.ev[0], ev_end = hp.ev[1];
  swa_status rc = cuda_ok(cudaEventRecord(ev_start, st), "cudaEventRecord");
  if (rc == SWA_OK) rc = cuda_ok(cudaStreamWaitEvent(hp.h2d, ev_start, 0), "cudaStreamWaitEvent");
  auto at = [](const void* base, size_t off) {
    return const_cast<char*>(static_cast<const char*>(base)) + off;
  };
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  for (int c = 0; rc == SWA_OK && c < nchunk; ++c) {
    const int b0 = (c / nsplit) * nseq, part = c % nsplit;
    const size_t rows = (size_t)nseq * T;                 // positions in the chunk
    const size_t hq0 = (size_t)part * Hq_c, hk0 = (size_t)part * Hkv_c;
    cudaEvent_t ev_in = hp.ev[2 + 2 * c], ev_c = hp.ev[3 + 2 * c];
    void* qc = at(q_d, c * q_chunk);
    void* kc = at(k_d, c * k_chunk);
    void* vc = at(v_d, c * k_chunk);
    void* oc = at(out_d, c * o_chunk);
    float* lc = lse_d ? reinterpret_cast<float*>(at(lse_d, c * l_chunk)) : nullptr;
    // rows of the chunk: positions b0*T .. (b0+nseq)*T - 1, heads hq0 .. hq0+Hq_c-1
    rc = cuda_ok(cudaMemcpy2DAsync(qc, q_row, at(q_h, b0 * (size_t)T * q_pitch + hq0 * D * ie),
                                   q_pitch, q_row, rows, h2d, hp.h2d),
                 "cudaMemcpy2DAsync(q)");
    if (rc == SWA_OK)
      rc = cuda_ok(cudaMemcpy2DAsync(kc, k_row, at(k_h, b0 * (size_t)T * k_pitch + hk0 * D * ie),
                                     k_pitch, k_row, rows, h2d, hp.h2d),
                   "cudaMemcpy2DAsync(k)");
    if (rc == SWA_OK)
      rc = cuda_ok(cudaMemcpy2DAsync(vc, k_row, at(v_h, b0 * (size_t)T * k_pitch + hk0 * D * ie),
                                     k_pitch, k_row, rows, h2d, hp.h2d),
                   "cudaMemcpy2DAsync(v)");
    if (rc == SWA_OK) rc = cuda_ok(cudaEventRecord(ev_in, hp.h2d), "cudaEventRecord");
    if (rc == SWA_OK) rc = cuda_ok(cudaStreamWaitEvent(st, ev_in, 0), "cudaStreamWaitEvent");
    if (rc == SWA_OK)
      rc = swa_sink_fwd_ex(qc, kc, vc, sink + hq0, oc, lc, nseq, T, Hq_c, Hkv_c, D, W, in_dtype,
                           out_dtype, stream);
    if (rc == SWA_OK) rc = cuda_ok(cudaEventRecord(ev_c, st), "cudaEventRecord");
    if (rc == SWA_OK) rc = cuda_ok(cudaStreamWaitEvent(hp.d2h, ev_c, 0), "cudaStreamWaitEvent");
    if (rc == SWA_OK)
      rc = cuda_ok(cudaMemcpy2DAsync(at(out_h, b0 * (size_t)T * o_pitch + hq0 * D * oe), o_pitch,
                                     oc, o_row, o_row, rows, d2h, hp.d2h),
                   "cudaMemcpy2DAsync(out)");
    // lse [B, Hq, T]: sequence b's heads hq0 .. are contiguous
    for (int b = b0; rc == SWA_OK && lse_d && b < b0 + nseq; ++b)
      rc = cuda_ok(cudaMemcpyAsync(at(lse_h, ((size_t)b * Hq + hq0) * T * 4),
                                   at(lc, (size_t)(b - b0) * Hq_c * T * 4), (size_t)Hq_c * T * 4,
                                   d2h, hp.d2h),
                   "cudaMemcpyAsync(lse)");
  }
  // later work on `stream` follows every copy enqueued above, even after an error
  const swa_status rc_end = cuda_ok(cudaEventRecord(ev_end, hp.d2h), "cudaEventRecord");
  const swa_status rc_wait =
      rc_end == SWA_OK ? cuda_ok(cudaStreamWaitEvent(st, ev_end, 0), "cudaStreamWaitEvent")
                       : rc_end;
  return rc != SWA_OK ? rc : rc_wait;
}

}  // extern "C"

// ---- host-memory prefill with library-owned staging (no allocation) -------
// Staging for swa_sink_fwd_host_static: one array per GPU, reserved when the
// library's module is loaded on that GPU and held until the process exits.
// Host code must not use the name as a device address; the address comes
// from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_host_staging[SWA_HOST_STATIC_BYTES];

namespace {
struct StagingAddr {
  bool ready = false;
  unsigned char* ptr = nullptr;
};
StagingAddr g_staging_addr[kMaxDevices];
std::mutex g_staging_mu;

// Device address of g_host_staging on `dev`, which must be the current device.
bool staging_base(int dev, unsigned char** base) {
  std::lock_guard<std::mutex> lk(g_staging_mu);
  StagingAddr& s = g_staging_addr[dev];
  if (!s.ready) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_host_staging);
    if (e != cudaSuccess) {
      set_cuda_error("cudaGetSymbolAddress(staging)", e);
      return false;
    }
    s.ptr = static_cast<unsigned char*>(p);
    s.ready = true;
  }
  *base = s.ptr;
  return true;
}

// a * b, saturated far above any staging size (sizes are positive ints).
unsigned long long mul_sat(unsigned long long a, unsigned long long b) {
  const unsigned long long cap = 1ull << 62;
  return (a != 0 && b > cap / a) ? cap : a * b;
}

unsigned long long round256(unsigned long long n) { return (n + 255ull) & ~255ull; }
}  // namespace

extern "C" {

swa_status swa_sink_fwd_host_static(const void* q_h, const void* k_h, const void* v_h,
                                    const float* sink, void* out_h, float* lse_h, int B, int T,
                                    int Hq, int Hkv, int D, int W, swa_dtype in_dtype,
                                    swa_dtype out_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!q_h || !k_h || !v_h || !out_h || !sink) return SWA_EINVAL;
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || Hq % Hkv) return SWA_EINVAL;
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return SWA_EINVAL;
  if (out_dtype != SWA_F32 && out_dtype != SWA_BF16) return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  // staging for q, k, v, out and lse, each at a 256-byte boundary
  const unsigned long long ie = in_dtype == SWA_BF16 ? 2 : 4, oe = out_dtype == SWA_BF16 ? 2 : 4;
  const unsigned long long pos = mul_sat((unsigned long long)B, (unsigned long long)T);
  const unsigned long long q_bytes = mul_sat(mul_sat(pos, (unsigned long long)Hq * D), ie);
  const unsigned long long k_bytes = mul_sat(mul_sat(pos, (unsigned long long)Hkv * D), ie);
  const unsigned long long o_bytes = mul_sat(mul_sat(pos, (unsigned long long)Hq * D), oe);
  const unsigned long long l_bytes = lse_h ? mul_sat(pos, (unsigned long long)Hq * 4) : 0;
  const unsigned long long off_k = round256(q_bytes), off_v = off_k + round256(k_bytes);
  const unsigned long long off_o = off_v + round256(k_bytes);
  const unsigned long long off_l = off_o + round256(o_bytes);
  const unsigned long long need = off_l + round256(l_bytes);
  if (need > (unsigned long long)SWA_HOST_STATIC_BYTES) {
    snprintf(g_last_error, sizeof g_last_error,
             "swa_sink_fwd_host_static: these sizes need %llu bytes of staging; the library's "
             "static staging holds %llu (SWA_HOST_STATIC_BYTES)",
             need, (unsigned long long)SWA_HOST_STATIC_BYTES);
    return SWA_EUNSUPPORTED;
  }
  int dev;
  if (!current_device(&dev)) return SWA_ECUDA;
  unsigned char* base = nullptr;
  if (!staging_base(dev, &base)) return SWA_ECUDA;
  // Every byte the pipeline reads from the staging is written earlier in the
  // same call, so nothing left by an earlier call is ever read: no clearing.
  return swa_sink_fwd_host(q_h, k_h, v_h, sink, out_h, lse_h, base, base + off_k, base + off_v,
                           base + off_o, lse_h ? reinterpret_cast<float*>(base + off_l) : nullptr,
                           B, T, Hq, Hkv, D, W, in_dtype, out_dtype, stream);
}

swa_status swa_sink_decode(const void* q, const void* k_ring, const void* v_ring,
                           const int64_t* pos, const float* sink, float* out, float* lse, int B,
                           int Hq, int Hkv, int D, int W, swa_dtype in_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!q || !k_ring || !v_ring || !pos || !sink || !out) return SWA_EINVAL;
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || Hq % Hkv) return SWA_EINVAL;
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(q) || !aligned16(k_ring) || !aligned16(v_ring) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (reinterpret_cast<uintptr_t>(pos) & 7u))
    return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  const int esz = in_dtype == SWA_F32 ? 4 : 2;
  if (2LL * W * D * esz > swa::kDecodeMaxRingBytes) return SWA_EUNSUPPORTED;
  if ((long long)B * Hkv > 0x7fffffffLL) return SWA_EUNSUPPORTED;
  int dev;
  if (!current_device(&dev)) return SWA_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (decode_tc_applies(Hq, Hkv, D, W, in_dtype))
    return launch_decode_tc(q, k_ring, v_ring, pos, sink, out, lse, B, Hq, Hkv, D, st, dev);
  if (in_dtype == SWA_F32) {
    if (D == 64)
      return launch_decode_g<float, 64>(q, k_ring, v_ring, pos, sink, out, lse, B, Hq, Hkv, W, st, dev);
    return launch_decode_g<float, 128>(q, k_ring, v_ring, pos, sink, out, lse, B, Hq, Hkv, W, st, dev);
  }
  if (D == 64)
    return launch_decode_g<__nv_bfloat16, 64>(q, k_ring, v_ring, pos, sink, out, lse, B, Hq, Hkv, W, st, dev);
  return launch_decode_g<__nv_bfloat16, 128>(q, k_ring, v_ring, pos, sink, out, lse, B, Hq, Hkv, W, st, dev);
}

swa_status swa_ring_append(const void* k_new, const void* v_new, void* k_ring, void* v_ring,
                           const int64_t* pos, int B, int Hkv, int D, int W, swa_dtype dtype,
                           void* stream) {
  g_last_error[0] = '\0';
  if (!k_new || !v_new || !k_ring || !v_ring || !pos) return SWA_EINVAL;
  if (B < 1 || Hkv < 1 || D < 1 || W < 1) return SWA_EINVAL;
  if (dtype != SWA_F32 && dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_ring) || !aligned16(v_ring) ||
      (reinterpret_cast<uintptr_t>(pos) & 7u))
    return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int esz = dtype == SWA_F32 ? 4 : 2;
  const long long total = (long long)B * Hkv * (D * esz / 16);
  const long long blocks_ll = (total + 255) / 256;
  const unsigned blocks = (unsigned)(blocks_ll < 4096 ? blocks_ll : 4096);
  if (dtype == SWA_F32)
    swa::ring_append_kernel<float><<<blocks, 256, 0, st>>>(
        static_cast<const float*>(k_new), static_cast<const float*>(v_new),
        static_cast<float*>(k_ring), static_cast<float*>(v_ring), pos, B, Hkv, D, W);
  else
    swa::ring_append_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
        static_cast<__nv_bfloat16*>(k_ring), static_cast<__nv_bfloat16*>(v_ring), pos, B, Hkv,
        D, W);
  return check_launch("ring_append_kernel");
}

swa_status swa_sink_verify(const void* q, const void* k_new, const void* v_new,
                           const void* k_ring, const void* v_ring, const int64_t* pos,
                           const float* sink, float* out, float* lse, int B, int L, int Hq,
                           int Hkv, int D, int W, swa_dtype in_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!q || !k_new || !v_new || !k_ring || !v_ring || !pos || !sink || !out) return SWA_EINVAL;
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || Hq % Hkv) return SWA_EINVAL;
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_ring) ||
      !aligned16(v_ring) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (reinterpret_cast<uintptr_t>(pos) & 7u))
    return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  if (L > kVerifyMaxL) return SWA_EUNSUPPORTED;
  const int esz = in_dtype == SWA_F32 ? 4 : 2;
  if (2LL * W * D * esz > swa::kDecodeMaxRingBytes) return SWA_EUNSUPPORTED;
  const long long rows = (long long)B * L * Hq;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffffLL) return SWA_EUNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (verify_tc_applies(L, Hq, Hkv, D, W, in_dtype))
    return launch_verify_tc(q, k_new, v_new, k_ring, v_ring, pos, sink, out, lse, B, L, Hq, Hkv, D,
                            st);
  const float scale = (float)(1.0 / std::sqrt((double)D));
#define SWA_VERIFY_LAUNCH(T, DD)                                                              \
  swa::verify_simt_kernel<T, DD><<<(unsigned)blocks, 256, 0, st>>>(                         \
      static_cast<const T*>(q), static_cast<const T*>(k_new), static_cast<const T*>(v_new), \
      static_cast<const T*>(k_ring), static_cast<const T*>(v_ring), pos, sink, out, lse, B,   \
      L, Hq, Hkv, W, scale)
  if (in_dtype == SWA_F32) {
    if (D == 64) SWA_VERIFY_LAUNCH(float, 64);
    else SWA_VERIFY_LAUNCH(float, 128);
  } else {
    if (D == 64) SWA_VERIFY_LAUNCH(__nv_bfloat16, 64);
    else SWA_VERIFY_LAUNCH(__nv_bfloat16, 128);
  }
#undef SWA_VERIFY_LAUNCH
  return check_launch("verify_simt_kernel");
}

static bool rope_args_ok(int D, int rot_dim, double theta) {
  return rot_dim >= 2 && rot_dim <= D && rot_dim % 2 == 0 && rot_dim / 2 <= swa::kRopeMaxHalf &&
         theta > 0.0 && std::isfinite(theta);
}

// f_i = theta^(-2 i / rot_dim) in fp64, the table the RoPE kernels read
static swa::RopeFreq rope_freq(int rot_dim, double theta) {
  swa::RopeFreq fr;
  for (int i = 0; i < swa::kRopeMaxHalf; ++i)
    fr.f[i] = i < rot_dim / 2 ? std::pow(theta, -2.0 * i / rot_dim) : 0.0;
  return fr;
}

swa_status swa_rope(void* x, const int64_t* pos0, int B, int T, int H, int D, int rot_dim,
                    double theta, swa_dtype dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!x || !pos0) return SWA_EINVAL;
  if (B < 1 || T < 1 || H < 1 || D < 1) return SWA_EINVAL;
  if ((long long)H * D > (1LL << 30)) return SWA_EUNSUPPORTED;   // per-token counts fit an int
  if (dtype != SWA_F32 && dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(pos0) & 7u)) return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  if (!rope_args_ok(D, rot_dim, theta)) return SWA_EINVAL;
  const long long ntok = (long long)B * T;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const swa::RopeFreq fr = rope_freq(rot_dim, theta);
  const int half = rot_dim / 2;
  const int V = dtype == SWA_F32 ? 4 : 8;
  const int vec = half % V == 0;   // whole 16-byte chunks
  // tokens per block: enough that a token's chunk tasks (H x half/V) fill the
  // block's threads at least once
  const int per_tok = H * (half / V);
  const int tpb = !vec ? 1
                       : (per_tok >= swa::kRopeThreads ? 1
                                                       : std::min(swa::kRopeMaxTok,
                                                                  swa::kRopeThreads / per_tok));
  const long long nblk = (ntok + tpb - 1) / tpb;
  const unsigned grid = (unsigned)(nblk < 65536 ? nblk : 65536);
  if (dtype == SWA_F32)
    swa::rope_inplace_kernel<float><<<grid, swa::kRopeThreads, 0, st>>>(
        static_cast<float*>(x), pos0, B, T, H, D, half, vec, tpb, fr);
  else
    swa::rope_inplace_kernel<__nv_bfloat16><<<grid, swa::kRopeThreads, 0, st>>>(
        static_cast<__nv_bfloat16*>(x), pos0, B, T, H, D, half, vec, tpb, fr);
  return check_launch("rope_inplace_kernel");
}

swa_status swa_rope_append(const void* q_in, const void* k_in, const void* v_in, void* q_out,
                           void* k_ring, void* v_ring, const int64_t* pos, int B, int Hq,
                           int Hkv, int D, int W, int rot_dim, double theta, swa_dtype dtype,
                           void* stream) {
  g_last_error[0] = '\0';
  if (!q_in || !k_in || !v_in || !q_out || !k_ring || !v_ring || !pos) return SWA_EINVAL;
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1) return SWA_EINVAL;
  if (dtype != SWA_F32 && dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(q_in) || !aligned16(k_in) || !aligned16(v_in) || !aligned16(q_out) ||
      !aligned16(k_ring) || !aligned16(v_ring) || (reinterpret_cast<uintptr_t>(pos) & 7u))
    return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  if (!rope_args_ok(D, rot_dim, theta)) return SWA_EINVAL;
  if ((long long)Hq + 2LL * Hkv > (1LL << 20)) return SWA_EUNSUPPORTED;   // task counts fit an int
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const swa::RopeFreq fr = rope_freq(rot_dim, theta);
  // 16-byte chunks when the rotated half is a whole number of them (every
  // buffer is 16-byte aligned and D is 64 or 128); a token's chunk tasks are
  // shared by S blocks of kRopeThreads threads
  const int half = rot_dim / 2;
  const int V = dtype == SWA_F32 ? 4 : 8;
  const int vec = half % V == 0;
  const int ntask = vec ? swa::rope_append_tasks(Hq, Hkv, D, half, V, q_in != q_out).total() : 0;
  const dim3 grid((unsigned)B, vec ? (unsigned)((ntask + swa::kRopeThreads - 1) / swa::kRopeThreads)
                                   : 1u);
  if (dtype == SWA_F32)
    swa::rope_append_kernel<float><<<grid, swa::kRopeThreads, 0, st>>>(
        static_cast<const float*>(q_in), static_cast<const float*>(k_in),
        static_cast<const float*>(v_in), static_cast<float*>(q_out), static_cast<float*>(k_ring),
        static_cast<float*>(v_ring), pos, Hq, Hkv, D, W, half, vec, fr);
  else
    swa::rope_append_kernel<__nv_bfloat16><<<grid, swa::kRopeThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(q_in), static_cast<const __nv_bfloat16*>(k_in),
        static_cast<const __nv_bfloat16*>(v_in), static_cast<__nv_bfloat16*>(q_out),
        static_cast<__nv_bfloat16*>(k_ring), static_cast<__nv_bfloat16*>(v_ring), pos, Hq, Hkv,
        D, W, half, vec, fr);
  return check_launch("rope_append_kernel");
}

swa_status swa_sink_fwd_scores(const void* q, const void* k, const void* v, const float* sink,
                               void* out, float* lse, float* blockmax, int B, int T, int Hq,
                               int Hkv, int D, int W, swa_dtype in_dtype, swa_dtype out_dtype,
                               void* stream) {
  g_last_error[0] = '\0';
  if (!q || !k || !v || !sink || !out || !blockmax) return SWA_EINVAL;
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || W < 1 || Hq % Hkv) return SWA_EINVAL;
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return SWA_EINVAL;
  if (out_dtype != SWA_F32 && out_dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (reinterpret_cast<uintptr_t>(blockmax) & 3u))
    return SWA_EINVAL;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  if (!(in_dtype == SWA_BF16 && Hq == Hkv * swa::tcglobal::kG)) {
    set_error_text("block scores come from the tensor-core global kernel (bf16, 8 heads per kv head)");
    return SWA_EUNSUPPORTED;
  }
  return launch_tc_global(q, k, v, sink, out, lse, B, T, Hq, Hkv, D, W, out_dtype == SWA_BF16,
                          static_cast<cudaStream_t>(stream), blockmax);
}

swa_status swa_topk_blocks(const float* scores, int* idx, int B, int T, int Hkv, int QB,
                           int topk, void* stream) {
  g_last_error[0] = '\0';
  if (!scores || !idx) return SWA_EINVAL;
  if (B < 1 || T < 1 || Hkv < 1 || QB < 4 || QB % 4 || 128 % QB || topk < 1) return SWA_EINVAL;
  if ((reinterpret_cast<uintptr_t>(scores) & 3u) || (reinterpret_cast<uintptr_t>(idx) & 3u))
    return SWA_EINVAL;
  const long long nkb = (T + 127LL) / 128;
  if (nkb > swa::kTopkMaxBlocks || topk > swa::kTopkMax) return SWA_EUNSUPPORTED;
  const long long units = (long long)B * Hkv * ((T + QB - 1LL) / QB);
  const long long blocks = (units + swa::kTopkWarps - 1) / swa::kTopkWarps;
  if (blocks > 0x7fffffffLL) return SWA_EUNSUPPORTED;
  const size_t smem = (size_t)swa::kTopkWarps * (nkb * 4 + ((nkb + 31) / 32) * 4);
  int dev;
  if (!current_device(&dev)) return SWA_ECUDA;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].topk_attr) {
      const int most = swa::kTopkWarps * (swa::kTopkMaxBlocks * 4 + swa::kTopkMaxBlocks / 8);
      cudaError_t e = cudaFuncSetAttribute(swa::topk_blocks_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, most);
      if (e != cudaSuccess) {
        set_cuda_error("cudaFuncSetAttribute(topk_blocks_kernel)", e);
        return SWA_ECUDA;
      }
      g_dev[dev].topk_attr = true;
    }
  }
  swa::topk_blocks_kernel<<<(unsigned)blocks, swa::kTopkWarps * 32, smem,
                            static_cast<cudaStream_t>(stream)>>>(scores, idx, B, T, Hkv, QB,
                                                                 topk);
  return check_launch("topk_blocks_kernel");
}

swa_status swa_sink_sparse_fwd(const void* q, const void* k, const void* v, const float* sink,
                               const int* idx, void* out, float* lse, int B, int T, int Hq,
                               int Hkv, int D, int QB, int topk, swa_dtype in_dtype,
                               swa_dtype out_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (!q || !k || !v || !sink || !idx || !out) return SWA_EINVAL;
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv || topk < 1) return SWA_EINVAL;
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return SWA_EINVAL;
  if (out_dtype != SWA_F32 && out_dtype != SWA_BF16) return SWA_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (lse && !aligned16(lse)) || (reinterpret_cast<uintptr_t>(idx) & 3u))
    return SWA_EINVAL;
  if (QB != 32 && QB != 64 && QB != 128) return SWA_EUNSUPPORTED;
  if (D != 64 && D != 128) return SWA_EUNSUPPORTED;
  if (!(in_dtype == SWA_BF16 && Hq == Hkv * swa::tcglobal::kG)) {
    set_error_text("sparse attention runs on the tensor-core global kernel (bf16, 8 heads per kv head)");
    return SWA_EUNSUPPORTED;
  }
  // causal over the selected blocks: no window lower bound
  return launch_tc_global(q, k, v, sink, out, lse, B, T, Hq, Hkv, D, T, out_dtype == SWA_BF16,
                          static_cast<cudaStream_t>(stream), nullptr, idx, QB, topk);
}

const char* swa_sink_verify_path(int B, int L, int Hq, int Hkv, int D, int W, swa_dtype in_dtype) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || W < 1 || Hq % Hkv) return "invalid";
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return "invalid";
  if (D != 64 && D != 128) return "invalid";
  if (L > kVerifyMaxL) return "invalid";
  const int esz = in_dtype == SWA_F32 ? 4 : 2;
  if (2LL * W * D * esz > swa::kDecodeMaxRingBytes) return "invalid";
  return verify_tc_applies(L, Hq, Hkv, D, W, in_dtype) ? "tc_verify" : "simt_verify";
}

const char* swa_sink_fwd_path(int B, int T, int Hq, int Hkv, int D, int W, swa_dtype in_dtype) {
  switch (select_fwd(B, T, Hq, Hkv, D, W, in_dtype)) {
    case kPathTcSwa: return "tc_swa";
    case kPathTcGlobal: return "tc_global";
    case kPathSimt: return "simt";
    default: return "invalid";
  }
}

const char* swa_sink_decode_path(int B, int Hq, int Hkv, int D, int W, swa_dtype in_dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1 || W < 1 || Hq % Hkv) return "invalid";
  if (in_dtype != SWA_F32 && in_dtype != SWA_BF16) return "invalid";
  if (D != 64 && D != 128) return "invalid";
  const int esz = in_dtype == SWA_F32 ? 4 : 2;
  if (2LL * W * D * esz > swa::kDecodeMaxRingBytes) return "invalid";
  return decode_tc_applies(Hq, Hkv, D, W, in_dtype) ? "tc_decode" : "simt_decode";
}

const char* swa_status_str(swa_status s) {
  switch (s) {
    case SWA_OK: return "ok";
    case SWA_EINVAL: return "invalid argument";
    case SWA_EUNSUPPORTED: return "unsupported configuration";
    case SWA_ECUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* swa_last_error(void) { return g_last_error; }

int swa_device_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    set_cuda_error("cudaDeviceSynchronize", e);
    return SWA_ECUDA;
  }
  unsigned int v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, swa::g_dev_error, sizeof v);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(swa::g_dev_error, &zero, sizeof zero);
  if (e != cudaSuccess) {
    set_cuda_error("device error word", e);
    return SWA_ECUDA;
  }
  return (int)v;
}

swa_status swa_test_withhold_loads(int cta) {
  g_last_error[0] = '\0';
  if (cta < -1) return SWA_EINVAL;
  g_withhold_cta = cta;
  return SWA_OK;
}

int swa_version(void) { return 100; }

}  // extern "C"
