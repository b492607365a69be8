// The C ABI of include/mi_block.h: argument validation, workspace planning, TMA descriptors and
// the launch sequence of a block forward and of a guided denoising step.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/mi_block.h"
#include "mi_internal.h"

namespace {

thread_local char g_err[512] = "";

mi_status fail(mi_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

mi_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MI_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MI_CUDA(call, what)                     \
  do {                                          \
    cudaError_t e_ = (call);                    \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Device error flag: kernels record the first pipeline timeout here.
__device__ int g_dev_err = 0;

struct DeviceInfo {
  bool ready = false;
  int* err = nullptr;
  int num_sms = 0;
  bool sm103 = false;
};
DeviceInfo g_dev[mi::kMaxDevices];
std::mutex g_dev_mu;

mi_status device_info(DeviceInfo** out) {
  int dev = 0;
  MI_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= mi::kMaxDevices) return fail(MI_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    MI_CUDA(cudaGetDeviceProperties(&prop, dev), "cudaGetDeviceProperties");
    d.sm103 = prop.major == 10 && prop.minor == 3;
    d.num_sms = prop.multiProcessorCount;
    void* p = nullptr;
    MI_CUDA(cudaGetSymbolAddress(&p, g_dev_err), "cudaGetSymbolAddress(error flag)");
    d.err = static_cast<int*>(p);
    d.ready = true;
  }
  *out = &d;
  return MI_OK;
}

mi_status require_sm103(DeviceInfo** out) {
  mi_status st = device_info(out);
  if (st != MI_OK) return st;
  if (!(*out)->sm103) return fail(MI_ERR_UNSUPPORTED, "the kernels are built for sm_103a (GB300) only");
  return MI_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using bf16 = __nv_bfloat16;

inline const bf16* cb(const void* p) { return static_cast<const bf16*>(p); }
inline bf16* mb(void* p) { return static_cast<bf16*>(p); }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
            const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                  reinterpret_cast<const cuuint64_t*>(dims), reinterpret_cast<const cuuint64_t*>(strides_bytes),
                  reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

namespace mi {

bool encode_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                    uint32_t box_inner, uint32_t box_rows) {
  const uint64_t dims[2] = {inner, rows};
  const uint64_t str[1] = {row_stride_bytes};
  const uint32_t box[2] = {box_inner, box_rows};
  return encode(m, base, 2, dims, str, box);
}

bool encode_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                    uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t str[2] = {s1_bytes, s2_bytes};
  const uint32_t box[3] = {b0, b1, b2};
  return encode(m, base, 3, dims, str, box);
}

bool encode_4d_bf16(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                    const uint32_t box[4]) {
  return encode(m, base, 4, dims, strides_bytes, box);
}

}  // namespace mi

// ------------------------------------------------------------------------------ GEMM helper
namespace {

// Every W operand map has 128-row boxes: the one-CTA GEMM loads a 256-row W tile as two boxes and
// each CTA of a pair loads one.
constexpr int kWBox = 128;

// A operand map: [rows, k] row-major, box 64 x 128.
bool map_a(CUtensorMap* m, const void* a, int rows, int k) {
  return mi::encode_2d_bf16(m, a, (uint64_t)k, (uint64_t)rows, (uint64_t)k * 2, 64, 128);
}

// W operand map: [rows, k] row-major, box 64 x box_rows.
bool map_w(CUtensorMap* m, const void* w, int rows, int k, int box_rows) {
  return mi::encode_2d_bf16(m, w, (uint64_t)k, (uint64_t)rows, (uint64_t)k * 2, 64, (uint32_t)box_rows);
}

mi_status check_gemm_shape(int m, int n, int k, int epi) {
  if (m <= 0 || n <= 0 || k <= 0) return fail(MI_ERR_INVALID_ARG, "gemm: m, n, k must be positive (%d, %d, %d)", m, n, k);
  if (k % 64 != 0) return fail(MI_ERR_UNSUPPORTED, "gemm: k=%d must be a multiple of 64", k);
  if (n % 8 != 0) return fail(MI_ERR_UNSUPPORTED, "gemm: n=%d must be a multiple of 8", n);
  if (epi == mi::EPI_SILU_GATE && n % 128 != 0)
    return fail(MI_ERR_UNSUPPORTED, "gemm+silu: inter=%d must be a multiple of 128", n);
  return MI_OK;
}

mi_status run_gemm(const DeviceInfo* dev, int epi, const CUtensorMap& ta, const CUtensorMap& tb, const mi::GemmArgs& ga,
                   cudaStream_t s) {
  cudaError_t e = mi::gemm_launch(epi, ta, tb, ga, dev->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
  return MI_OK;
}

mi::GemmArgs gemm_args(int m, int n, int k, void* c, int* err) {
  mi::GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.M = m;
  g.N = n;
  g.K = k;
  g.C = mb(c);
  g.ldc = n;
  g.seq = 1;
  g.err = err;
  return g;
}

}  // namespace

// ------------------------------------------------------------------------------ block
struct mi_block {
  mi_block_desc d;
  CUtensorMap tm_wqkv, tm_wo, tm_wgu, tm_wd;
  int dev;
  int num_sms;
};

struct WsLayout {
  size_t off[11];
  size_t bytes[11];
  bool present[11];
  size_t sk_off, sk_bytes;  // stream-K scratch of the out and down projections (0 bytes: not used)
  size_t at_off, at_bytes;  // attention scratch: arrival counters, then the partial results (0: none)
  size_t total;
};

static WsLayout plan_ws(const mi_block_desc& d, int batch, int seq, int num_sms) {
  WsLayout w;
  const size_t R = (size_t)batch * seq;
  const size_t H = d.hidden, I = d.mlp_inter;
  const size_t sizes[11] = {R * H, R * 3 * H, R * H, R * H, R * H, R * H, R * H, R * H, R * 2 * I, R * I, R * H};
  const bool fused = d.fuse_epilogues != 0;
  size_t cur = 0;
  for (int i = 0; i < 11; ++i) {
    const bool pres = !(fused && (i == MI_T_A || i == MI_T_GU || i == MI_T_DN));
    w.present[i] = pres;
    w.bytes[i] = pres ? sizes[i] * 2 : 0;
    w.off[i] = cur;
    if (pres) cur = align_up(cur + w.bytes[i], 1024);
  }
  // the out (K = H) and down (K = I) projections run one after the other and share the scratch
  const int Ri = batch * seq;
  const size_t sk_o = mi::gemm_sk_scratch_bytes(mi::EPI_GATED_RESIDUAL, Ri, (int)H, (int)H, num_sms);
  const size_t sk_d = mi::gemm_sk_scratch_bytes(mi::EPI_GATED_RESIDUAL, Ri, (int)H, (int)I, num_sms);
  w.sk_bytes = sk_o > sk_d ? sk_o : sk_d;
  w.sk_off = cur;
  cur = align_up(cur + w.sk_bytes, 1024);
  w.at_bytes = mi::attention_scratch_bytes(batch, seq, d.n_heads, num_sms);
  w.at_off = cur;
  cur = align_up(cur + w.at_bytes, 1024);
  w.total = cur;
  return w;
}

static mi_status check_desc(const mi_block_desc* d) {
  if (!d) return fail(MI_ERR_INVALID_ARG, "null descriptor");
  if (d->head_dim != 128) return fail(MI_ERR_UNSUPPORTED, "head_dim=%d: only 128 is supported", d->head_dim);
  if (d->n_heads <= 0 || d->hidden != d->n_heads * 128)
    return fail(MI_ERR_INVALID_ARG, "hidden=%d must equal n_heads*128 (n_heads=%d)", d->hidden, d->n_heads);
  if (d->hidden % 256 != 0 || d->hidden > 4096)
    return fail(MI_ERR_UNSUPPORTED, "hidden=%d must be a multiple of 256 and at most 4096", d->hidden);
  if (d->mlp_inter <= 0 || d->mlp_inter % 128 != 0)
    return fail(MI_ERR_UNSUPPORTED, "mlp_inter=%d must be a positive multiple of 128", d->mlp_inter);
  if (!(d->eps >= 0.0f)) return fail(MI_ERR_INVALID_ARG, "eps must be >= 0");
  const void* w[6] = {d->w_qkv, d->w_o, d->w_gu, d->w_d, d->q_norm_w, d->k_norm_w};
  const char* names[6] = {"w_qkv", "w_o", "w_gu", "w_d", "q_norm_w", "k_norm_w"};
  for (int i = 0; i < 6; ++i) {
    if (!w[i]) return fail(MI_ERR_INVALID_ARG, "weight %s is null", names[i]);
    if (!aligned16(w[i])) return fail(MI_ERR_INVALID_ARG, "weight %s is not 16-byte aligned", names[i]);
  }
  return MI_OK;
}

static mi_status check_layout(const mi_seq_layout* L, int* seq) {
  if (!L) return fail(MI_ERR_INVALID_ARG, "null layout");
  if (L->batch <= 0 || L->text_pad < 0 || L->grid_h < 0 || L->grid_w < 0)
    return fail(MI_ERR_INVALID_ARG, "bad layout (batch=%d text_pad=%d grid=%dx%d)", L->batch, L->text_pad,
                L->grid_h, L->grid_w);
  const long long S = (long long)L->text_pad + (long long)L->grid_h * L->grid_w;
  if (S <= 0 || S > (1 << 20)) return fail(MI_ERR_INVALID_ARG, "sequence length %lld out of range", S);
  *seq = (int)S;
  return MI_OK;
}

static mi_status block_forward_impl(mi_block* blk, int batch, int S, const void* x, void* y, const void* mod,
                                    const float* cosv, const float* sinv, int rope_bstride, const uint8_t* key_mask,
                                    void* ws, size_t ws_bytes, cudaStream_t s, const DeviceInfo* dev) {
  const mi_block_desc& d = blk->d;
  const int H = d.hidden, I = d.mlp_inter, nh = d.n_heads;
  const int R = batch * S;
  const WsLayout w = plan_ws(d, batch, S, blk->num_sms);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(MI_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  if (ws_bytes < w.total) return fail(MI_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, w.total);
  uint8_t* base = static_cast<uint8_t*>(ws);
  bf16* h = mb(base + w.off[MI_T_H]);
  bf16* qkv = mb(base + w.off[MI_T_QKV]);
  bf16* qp = mb(base + w.off[MI_T_QP]);
  bf16* kp = mb(base + w.off[MI_T_KP]);
  bf16* o = mb(base + w.off[MI_T_O]);
  bf16* a = mb(base + w.off[MI_T_A]);
  bf16* x1 = mb(base + w.off[MI_T_X1]);
  bf16* h2 = mb(base + w.off[MI_T_H2]);
  bf16* gu = mb(base + w.off[MI_T_GU]);
  bf16* m = mb(base + w.off[MI_T_M]);
  bf16* dn = mb(base + w.off[MI_T_DN]);
  void* sk = w.sk_bytes ? static_cast<void*>(base + w.sk_off) : nullptr;
  int* at_count = w.at_bytes ? reinterpret_cast<int*>(base + w.at_off) : nullptr;
  float* at_part = w.at_bytes ? reinterpret_cast<float*>(base + w.at_off + mi::attention_count_bytes(batch, S, nh))
                              : nullptr;
  const int at_count_n = w.at_bytes ? (int)(mi::attention_count_bytes(batch, S, nh) / sizeof(int)) : 0;
  const bf16* md = cb(mod);
  const int mbs = 6 * H;  // batch stride of the modulation rows
  cudaError_t e;

  // activation operand maps of this call
  CUtensorMap tm_h, tm_o, tm_h2, tm_m, tq, tk, tv;
  if (!map_a(&tm_h, h, R, H) || !map_a(&tm_o, o, R, H) || !map_a(&tm_h2, h2, R, H) || !map_a(&tm_m, m, R, I))
    return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (activation operands)");
  if (!mi::encode_3d_bf16(&tq, qp, 128, (uint64_t)S, (uint64_t)batch * nh, 256, (uint64_t)S * 256, 64, 128, 1) ||
      !mi::encode_3d_bf16(&tk, kp, 128, (uint64_t)S, (uint64_t)batch * nh, 256, (uint64_t)S * 256, 64, 128, 1))
    return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (q/k)");
  {
    const uint64_t dims[4] = {128, (uint64_t)nh, (uint64_t)S, (uint64_t)batch};
    const uint64_t str[3] = {256, (uint64_t)3 * H * 2, (uint64_t)S * 3 * H * 2};
    const uint32_t box[4] = {64, 1, 128, 1};
    if (!mi::encode_4d_bf16(&tv, qkv + 2 * H, dims, str, box)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (v)");
  }

  // 1. modulated RMSNorm #1 (it also clears the attention's arrival counters)
  e = mi::mod_rmsnorm_launch(cb(x), md + 0 * H, md + 1 * H, mbs, h, R, S, H, d.eps, dev->err, s, at_count, at_count_n);
  if (e != cudaSuccess) return cuda_fail(e, "mod_rmsnorm");
  // 2-3. QKV projection; q/k RMSNorm + rotary, packed per head (fused into the projection's epilogue,
  // or a separate kernel when epilogues are not fused)
  if (d.fuse_epilogues) {
    mi::GemmArgs g = gemm_args(R, 3 * H, H, qkv, dev->err);
    g.seq = S;
    g.qp = qp;
    g.kp = kp;
    g.wq = cb(d.q_norm_w);
    g.wk = cb(d.k_norm_w);
    g.rope_cos = cosv;
    g.rope_sin = sinv;
    g.rope_bstride = rope_bstride;
    g.hidden = H;
    g.heads = nh;
    g.eps = d.eps;
    mi_status st = run_gemm(dev, mi::EPI_QKV_ROPE, tm_h, blk->tm_wqkv, g, s);
    if (st != MI_OK) return st;
  } else {
    mi::GemmArgs g = gemm_args(R, 3 * H, H, qkv, dev->err);
    mi_status st = run_gemm(dev, mi::EPI_STORE, tm_h, blk->tm_wqkv, g, s);
    if (st != MI_OK) return st;
    e = mi::qk_norm_rope_launch(qkv, cb(d.q_norm_w), cb(d.k_norm_w), cosv, sinv, rope_bstride, qp, kp, batch, S, nh,
                                d.eps, s);
    if (e != cudaSuccess) return cuda_fail(e, "qk_norm_rope");
  }
  // 4. attention
  {
    mi::AttnArgs aa;
    aa.batch = batch;
    aa.seq = S;
    aa.n_heads = nh;
    aa.key_mask = key_mask;
    aa.out = o;
    aa.scale_log2 = 1.4426950408889634f / sqrtf(128.0f);
    aa.err = dev->err;
    aa.part = at_part;
    aa.count = at_count;
    e = mi::attention_launch(tq, tk, tv, aa, blk->num_sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  }
  // 5. out projection + gated residual
  if (d.fuse_epilogues) {
    mi::GemmArgs g = gemm_args(R, H, H, x1, dev->err);
    g.sk_scratch = sk;
    g.resid = cb(x);
    g.ldr = H;
    g.gate = md + 2 * H;
    g.gate_bstride = mbs;
    g.seq = S;
    mi_status st = run_gemm(dev, mi::EPI_GATED_RESIDUAL, tm_o, blk->tm_wo, g, s);
    if (st != MI_OK) return st;
  } else {
    mi::GemmArgs g = gemm_args(R, H, H, a, dev->err);
    g.sk_scratch = sk;
    mi_status st = run_gemm(dev, mi::EPI_STORE, tm_o, blk->tm_wo, g, s);
    if (st != MI_OK) return st;
    e = mi::gated_add_launch(cb(x), a, md + 2 * H, mbs, x1, R, S, H, s);
    if (e != cudaSuccess) return cuda_fail(e, "gated_add");
  }
  // 6. modulated RMSNorm #2
  e = mi::mod_rmsnorm_launch(x1, md + 3 * H, md + 4 * H, mbs, h2, R, S, H, d.eps, dev->err, s);
  if (e != cudaSuccess) return cuda_fail(e, "mod_rmsnorm");
  // 7. gate/up projection + SiLU gate
  if (d.fuse_epilogues) {
    mi::GemmArgs g = gemm_args(R, I, H, m, dev->err);
    mi_status st = run_gemm(dev, mi::EPI_SILU_GATE, tm_h2, blk->tm_wgu, g, s);
    if (st != MI_OK) return st;
  } else {
    mi::GemmArgs g = gemm_args(R, 2 * I, H, gu, dev->err);
    mi_status st = run_gemm(dev, mi::EPI_STORE, tm_h2, blk->tm_wgu, g, s);
    if (st != MI_OK) return st;
    e = mi::silu_gate_launch(gu, m, R, I, s);
    if (e != cudaSuccess) return cuda_fail(e, "silu_gate");
  }
  // 8. down projection + gated residual
  if (d.fuse_epilogues) {
    mi::GemmArgs g = gemm_args(R, H, I, y, dev->err);
    g.sk_scratch = sk;
    g.resid = x1;
    g.ldr = H;
    g.gate = md + 5 * H;
    g.gate_bstride = mbs;
    g.seq = S;
    mi_status st = run_gemm(dev, mi::EPI_GATED_RESIDUAL, tm_m, blk->tm_wd, g, s);
    if (st != MI_OK) return st;
  } else {
    mi::GemmArgs g = gemm_args(R, H, I, dn, dev->err);
    g.sk_scratch = sk;
    mi_status st = run_gemm(dev, mi::EPI_STORE, tm_m, blk->tm_wd, g, s);
    if (st != MI_OK) return st;
    e = mi::gated_add_launch(x1, dn, md + 5 * H, mbs, mb(y), R, S, H, s);
    if (e != cudaSuccess) return cuda_fail(e, "gated_add");
  }
  return MI_OK;
}

extern "C" {

const char* mi_last_error(void) { return g_err; }

int mi_abi_version(void) { return MI_ABI_VERSION; }

mi_status mi_device_supported(void) {
  DeviceInfo* dev = nullptr;
  return require_sm103(&dev);
}

mi_status mi_device_error(int* code) {
  if (!code) return fail(MI_ERR_INVALID_ARG, "null code");
  DeviceInfo* dev = nullptr;
  mi_status st = device_info(&dev);
  if (st != MI_OK) return st;
  MI_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  int v = 0;
  MI_CUDA(cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(int)), "read device error flag");
  const int zero = 0;
  MI_CUDA(cudaMemcpyToSymbol(g_dev_err, &zero, sizeof(int)), "clear device error flag");
  *code = v;
  return MI_OK;
}

mi_status mi_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us <= 0 || limit_us > 1000000) return fail(MI_ERR_INVALID_ARG, "limit_us must be in (0, 1e6]");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaError_t e = mi::wait_timeout_selftest_launch(dev->err, (unsigned long long)limit_us * 1000ull,
                                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "wait self-test launch");
}

mi_status mi_block_init(mi_block** out, const mi_block_desc* desc) {
  if (!out) return fail(MI_ERR_INVALID_ARG, "null output pointer");
  *out = nullptr;
  mi_status st = check_desc(desc);
  if (st != MI_OK) return st;
  DeviceInfo* dev = nullptr;
  st = require_sm103(&dev);
  if (st != MI_OK) return st;
  mi_block* b = new (std::nothrow) mi_block;
  if (!b) return fail(MI_ERR_INVALID_ARG, "host allocation failed");
  b->d = *desc;
  b->num_sms = dev->num_sms;
  MI_CUDA(cudaGetDevice(&b->dev), "cudaGetDevice");
  const int H = desc->hidden, I = desc->mlp_inter;
  if (!map_w(&b->tm_wqkv, desc->w_qkv, 3 * H, H, kWBox) || !map_w(&b->tm_wo, desc->w_o, H, H, kWBox) ||
      !map_w(&b->tm_wgu, desc->w_gu, 2 * I, H, kWBox) || !map_w(&b->tm_wd, desc->w_d, H, I, kWBox)) {
    delete b;
    return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (weights)");
  }
  *out = b;
  return MI_OK;
}

void mi_block_destroy(mi_block* blk) { delete blk; }

mi_status mi_block_workspace_size(const mi_block* blk, int batch, int seq, size_t* bytes) {
  if (!blk || !bytes) return fail(MI_ERR_INVALID_ARG, "null argument");
  if (batch <= 0 || seq <= 0) return fail(MI_ERR_INVALID_ARG, "batch and seq must be positive");
  *bytes = plan_ws(blk->d, batch, seq, blk->num_sms).total;
  return MI_OK;
}

mi_status mi_block_tensor_offset(const mi_block* blk, int batch, int seq, int which, size_t* offset, size_t* bytes) {
  if (!blk || !offset || !bytes) return fail(MI_ERR_INVALID_ARG, "null argument");
  if (which < 0 || which > MI_T_DN) return fail(MI_ERR_INVALID_ARG, "unknown tensor %d", which);
  const WsLayout w = plan_ws(blk->d, batch, seq, blk->num_sms);
  if (!w.present[which]) return fail(MI_ERR_UNSUPPORTED, "tensor %d is not materialised with fused epilogues", which);
  *offset = w.off[which];
  *bytes = w.bytes[which];
  return MI_OK;
}

mi_status mi_block_forward(mi_block* blk, const mi_seq_layout* L, const void* x, void* y, const void* mod,
                           const float* rope_cos, const float* rope_sin, int rope_bstride, const uint8_t* key_mask,
                           void* ws, size_t ws_bytes, void* stream) {
  if (!blk) return fail(MI_ERR_INVALID_ARG, "null block");
  int S = 0;
  mi_status st = check_layout(L, &S);
  if (st != MI_OK) return st;
  if (!x || !y || !mod || !rope_cos || !rope_sin) return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(x) || !aligned16(y) || !aligned16(mod) || !aligned16(rope_cos) || !aligned16(rope_sin))
    return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (rope_bstride < 0 || rope_bstride % 4 != 0) return fail(MI_ERR_INVALID_ARG, "rope_bstride must be >= 0 and a multiple of 4");
  const size_t xb = (size_t)L->batch * S * blk->d.hidden * 2;
  const uint8_t* xs = static_cast<const uint8_t*>(x);
  const uint8_t* ys = static_cast<const uint8_t*>(y);
  if (x != y && xs < ys + xb && ys < xs + xb) return fail(MI_ERR_INVALID_ARG, "x and y overlap without being equal");
  DeviceInfo* dev = nullptr;
  st = require_sm103(&dev);
  if (st != MI_OK) return st;
  return block_forward_impl(blk, L->batch, S, x, y, mod, rope_cos, rope_sin, rope_bstride, key_mask, ws, ws_bytes,
                            static_cast<cudaStream_t>(stream), dev);
}

// ------------------------------------------------------------------------------ model / step
}  // extern "C"

struct mi_model {
  std::vector<mi_block*> blocks;
  int n_blocks, latent_ch, hidden;
  const void* w_in;
  const void* w_out;
  CUtensorMap tm_win, tm_wout;
};

struct StepLayout {
  size_t lat16, u, x, hf, vel, blk, total;
};

static StepLayout plan_step(const mi_model* m, int batch, int S, int n_img) {
  StepLayout l;
  const size_t H = m->hidden, C = m->latent_ch;
  size_t cur = 0;
  l.lat16 = cur;
  cur = align_up(cur + (size_t)n_img * C * 2, 1024);
  l.u = cur;
  cur = align_up(cur + (size_t)n_img * H * 2, 1024);
  l.x = cur;
  cur = align_up(cur + (size_t)batch * S * H * 2, 1024);
  l.hf = cur;
  cur = align_up(cur + (size_t)batch * n_img * H * 2, 1024);
  l.vel = cur;
  cur = align_up(cur + (size_t)batch * n_img * C * 4, 1024);
  l.blk = cur;
  cur += plan_ws(m->blocks[0]->d, batch, S, m->blocks[0]->num_sms).total;
  l.total = align_up(cur, 1024);
  return l;
}

extern "C" {

mi_status mi_model_init(mi_model** out, const mi_model_desc* desc) {
  if (!out || !desc) return fail(MI_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  if (desc->n_blocks <= 0 || !desc->blocks) return fail(MI_ERR_INVALID_ARG, "model needs at least one block");
  if (desc->latent_ch <= 0 || desc->latent_ch % 64 != 0)
    return fail(MI_ERR_UNSUPPORTED, "latent_ch=%d must be a positive multiple of 64", desc->latent_ch);
  if (!desc->w_in || !desc->w_out || !aligned16(desc->w_in) || !aligned16(desc->w_out))
    return fail(MI_ERR_INVALID_ARG, "w_in / w_out must be non-null and 16-byte aligned");
  mi_model* m = new (std::nothrow) mi_model;
  if (!m) return fail(MI_ERR_INVALID_ARG, "host allocation failed");
  m->n_blocks = desc->n_blocks;
  m->latent_ch = desc->latent_ch;
  m->hidden = desc->blocks[0].hidden;
  m->w_in = desc->w_in;
  m->w_out = desc->w_out;
  for (int i = 0; i < desc->n_blocks; ++i) {
    const mi_block_desc& bd = desc->blocks[i];
    if (bd.hidden != m->hidden || bd.mlp_inter != desc->blocks[0].mlp_inter || bd.n_heads != desc->blocks[0].n_heads) {
      mi_model_destroy(m);
      return fail(MI_ERR_INVALID_ARG, "block %d geometry differs from block 0", i);
    }
    mi_block* b = nullptr;
    mi_status st = mi_block_init(&b, &bd);
    if (st != MI_OK) {
      mi_model_destroy(m);
      return st;
    }
    m->blocks.push_back(b);
  }
  if (!map_w(&m->tm_win, m->w_in, m->hidden, m->latent_ch, kWBox) ||
      !map_w(&m->tm_wout, m->w_out, m->latent_ch, m->hidden, kWBox)) {
    mi_model_destroy(m);
    return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (embedders)");
  }
  *out = m;
  return MI_OK;
}

void mi_model_destroy(mi_model* model) {
  if (!model) return;
  for (mi_block* b : model->blocks) mi_block_destroy(b);
  delete model;
}

mi_status mi_model_workspace_size(const mi_model* model, const mi_seq_layout* L, size_t* bytes) {
  if (!model || !bytes) return fail(MI_ERR_INVALID_ARG, "null argument");
  int S = 0;
  mi_status st = check_layout(L, &S);
  if (st != MI_OK) return st;
  *bytes = plan_step(model, L->batch, S, L->grid_h * L->grid_w).total;
  return MI_OK;
}

mi_status mi_model_plan(const mi_model* model, const mi_seq_layout* layouts, int n, size_t budget_bytes,
                        size_t* bytes, uint8_t* served) {
  if (!model || !layouts || !bytes) return fail(MI_ERR_INVALID_ARG, "null argument");
  if (n < 1) return fail(MI_ERR_INVALID_ARG, "plan needs at least one layout (n=%d)", n);
  size_t most = 0;
  int n_served = 0;
  for (int i = 0; i < n; ++i) {
    int S = 0;
    mi_status st = check_layout(&layouts[i], &S);
    if (st != MI_OK) return st;
    const size_t need = plan_step(model, layouts[i].batch, S, layouts[i].grid_h * layouts[i].grid_w).total;
    const bool ok = need <= budget_bytes;
    if (served) served[i] = ok ? 1 : 0;
    if (ok) {
      ++n_served;
      if (need > most) most = need;
    }
  }
  *bytes = most;
  if (n_served == 0)
    return fail(MI_ERR_WORKSPACE, "out of device memory: none of the %d layouts fits in %zu bytes", n, budget_bytes);
  return MI_OK;
}

mi_status mi_denoise_step(mi_model* model, const mi_seq_layout* L, void* latent, const void* text_rows,
                          const void* mods, const void* mod_final, const float* rope_cos, const float* rope_sin,
                          int rope_bstride, const uint8_t* key_mask, float dt, float guidance,
                          const uint8_t* skip_neg, void* ws, size_t ws_bytes, void* stream) {
  if (!model) return fail(MI_ERR_INVALID_ARG, "null model");
  int S = 0;
  mi_status st = check_layout(L, &S);
  if (st != MI_OK) return st;
  if (L->batch > 2) return fail(MI_ERR_UNSUPPORTED, "a guided step takes batch 1 or 2 (prompt, negative)");
  if (!latent || !mods || !mod_final || !rope_cos || !rope_sin || (L->text_pad > 0 && !text_rows))
    return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(latent) || !aligned16(mods) || !aligned16(mod_final) || (text_rows && !aligned16(text_rows)))
    return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const int N = L->grid_h * L->grid_w;
  if (N <= 0) return fail(MI_ERR_INVALID_ARG, "a denoising step needs image tokens");
  const StepLayout sl = plan_step(model, L->batch, S, N);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(MI_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  if (ws_bytes < sl.total) return fail(MI_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, sl.total);
  DeviceInfo* dev = nullptr;
  st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = model->hidden, C = model->latent_ch, B = L->batch;
  uint8_t* base = static_cast<uint8_t*>(ws);
  bf16* u = mb(base + sl.u);
  bf16* x = mb(base + sl.x);
  bf16* hf = mb(base + sl.hf);
  bf16* lat16 = mb(base + sl.lat16);
  float* vel = reinterpret_cast<float*>(base + sl.vel);
  void* bws = base + sl.blk;
  const size_t bws_bytes = ws_bytes - sl.blk;
  cudaError_t e;

  // latent embedding u = bf16(latent) W_in^T, then x_b = [text_b ; u]
  e = mi::f32_to_bf16_launch(static_cast<const float*>(latent), lat16, (size_t)N * C, s);
  if (e != cudaSuccess) return cuda_fail(e, "latent cast");
  {
    CUtensorMap ta;
    if (!map_a(&ta, lat16, N, C)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (latent)");
    mi::GemmArgs g = gemm_args(N, H, C, u, dev->err);
    st = run_gemm(dev, mi::EPI_STORE, ta, model->tm_win, g, s);
    if (st != MI_OK) return st;
  }
  e = mi::assemble_seq_launch(cb(text_rows), u, x, B, L->text_pad, N, H, s);
  if (e != cudaSuccess) return cuda_fail(e, "assemble_seq");

  const bf16* md = cb(mods);
  for (int i = 0; i < model->n_blocks; ++i) {
    const bf16* mod_i = md + (size_t)i * B * 6 * H;
    const bool skip = skip_neg != nullptr && skip_neg[i] != 0 && B == 2;
    const int nb = skip ? 1 : B;  // the negative element (index 1) bypasses this block
    st = block_forward_impl(model->blocks[i], nb, S, x, x, mod_i, rope_cos, rope_sin, rope_bstride, key_mask, bws,
                            bws_bytes, s, dev);
    if (st != MI_OK) return st;
  }

  // velocity head on the image rows, guidance and the Euler update
  const bf16* mf = cb(mod_final);
  e = mi::mod_rmsnorm_rows_launch(x, mf + 0, mf + H, 2 * H, hf, B * N, N, S, L->text_pad, H,
                                  model->blocks[0]->d.eps, dev->err, s);
  if (e != cudaSuccess) return cuda_fail(e, "final norm");
  {
    CUtensorMap ta;
    if (!map_a(&ta, hf, B * N, H)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (final rows)");
    mi::GemmArgs g = gemm_args(B * N, C, H, vel, dev->err);  // fp32 velocities (ldc = C floats)
    st = run_gemm(dev, mi::EPI_STORE_F32, ta, model->tm_wout, g, s);
    if (st != MI_OK) return st;
  }
  e = mi::cfg_euler_launch(vel, static_cast<float*>(latent), N, C, dt, guidance, B, s);
  if (e != cudaSuccess) return cuda_fail(e, "cfg_euler");
  return MI_OK;
}

// ------------------------------------------------------------------------------ single kernels
mi_status mi_mod_rmsnorm(const void* x, const void* mod, int shift_row, int scale_row, void* out, int batch, int seq,
                         int hidden, float eps, void* stream) {
  if (!x || !mod || !out) return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(x) || !aligned16(mod) || !aligned16(out)) return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (batch <= 0 || seq <= 0) return fail(MI_ERR_INVALID_ARG, "batch and seq must be positive");
  if (hidden <= 0 || hidden % 256 != 0 || hidden > 4096)
    return fail(MI_ERR_UNSUPPORTED, "hidden=%d must be a multiple of 256 and at most 4096", hidden);
  if (shift_row < 0 || shift_row > 5 || scale_row < 0 || scale_row > 5) return fail(MI_ERR_INVALID_ARG, "mod rows are 0..5");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  const bf16* md = cb(mod);
  cudaError_t e = mi::mod_rmsnorm_launch(cb(x), md + (size_t)shift_row * hidden, md + (size_t)scale_row * hidden,
                                         6 * hidden, mb(out), batch * seq, seq, hidden, eps, dev->err,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "mod_rmsnorm");
}

static mi_status gemm_common(int epi, const void* a, const void* w, void* c, int m, int n, int k, const void* resid,
                             const void* mod, int gate_row, int seq, void* stream) {
  if (!a || !w || !c) return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(a) || !aligned16(w) || !aligned16(c) || (resid && !aligned16(resid)) || (mod && !aligned16(mod)))
    return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  mi_status st = check_gemm_shape(m, n, k, epi);
  if (st != MI_OK) return st;
  DeviceInfo* dev = nullptr;
  st = require_sm103(&dev);
  if (st != MI_OK) return st;
  CUtensorMap ta, tb;
  const int w_rows = epi == mi::EPI_SILU_GATE ? 2 * n : n;
  if (!map_a(&ta, a, m, k) || !map_w(&tb, w, w_rows, k, kWBox))
    return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed");
  mi::GemmArgs g = gemm_args(m, n, k, c, dev->err);
  if (epi == mi::EPI_GATED_RESIDUAL) {
    if (!resid || !mod) return fail(MI_ERR_INVALID_ARG, "null resid or mod");
    if (gate_row < 0 || gate_row > 5) return fail(MI_ERR_INVALID_ARG, "gate_row is 0..5");
    if (seq <= 0 || m % seq != 0) return fail(MI_ERR_INVALID_ARG, "m must be a multiple of seq");
    g.resid = cb(resid);
    g.ldr = n;
    g.gate = cb(mod) + (size_t)gate_row * n;
    g.gate_bstride = 6 * n;
    g.seq = seq;
  }
  return run_gemm(dev, epi, ta, tb, g, static_cast<cudaStream_t>(stream));
}

mi_status mi_gemm_bf16(const void* a, const void* w, void* c, int m, int n, int k, void* stream) {
  return gemm_common(mi::EPI_STORE, a, w, c, m, n, k, nullptr, nullptr, 0, 1, stream);
}

mi_status mi_gemm_bf16_gated_residual(const void* a, const void* w, const void* resid, const void* mod, int gate_row,
                                      void* out, int m, int n, int k, int seq, void* stream) {
  return gemm_common(mi::EPI_GATED_RESIDUAL, a, w, out, m, n, k, resid, mod, gate_row, seq, stream);
}

mi_status mi_gemm_bf16_silu_gate(const void* a, const void* w, void* m_out, int m, int inter, int k, void* stream) {
  return gemm_common(mi::EPI_SILU_GATE, a, w, m_out, m, inter, k, nullptr, nullptr, 0, 1, stream);
}

mi_status mi_gemm_bf16_qkv_rope(const void* a, const void* w_qkv, const void* q_norm_w, const void* k_norm_w,
                                const float* rope_cos, const float* rope_sin, int rope_bstride, void* qp, void* kp,
                                void* qkv_v, int batch, int seq, int n_heads, float eps, void* stream) {
  if (!a || !w_qkv || !q_norm_w || !k_norm_w || !rope_cos || !rope_sin || !qp || !kp || !qkv_v)
    return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(a) || !aligned16(w_qkv) || !aligned16(q_norm_w) || !aligned16(k_norm_w) || !aligned16(rope_cos) ||
      !aligned16(rope_sin) || !aligned16(qp) || !aligned16(kp) || !aligned16(qkv_v))
    return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (batch <= 0 || seq <= 0 || n_heads <= 0) return fail(MI_ERR_INVALID_ARG, "batch, seq, n_heads must be positive");
  const int H = n_heads * 128;
  if (H % 256 != 0) return fail(MI_ERR_UNSUPPORTED, "hidden=%d must be a multiple of 256", H);
  if (rope_bstride < 0 || rope_bstride % 4 != 0) return fail(MI_ERR_INVALID_ARG, "bad rope_bstride");
  const int m = batch * seq;
  mi_status st = check_gemm_shape(m, 3 * H, H, mi::EPI_QKV_ROPE);
  if (st != MI_OK) return st;
  DeviceInfo* dev = nullptr;
  st = require_sm103(&dev);
  if (st != MI_OK) return st;
  CUtensorMap ta, tb;
  if (!map_a(&ta, a, m, H) || !map_w(&tb, w_qkv, 3 * H, H, kWBox)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed");
  mi::GemmArgs g = gemm_args(m, 3 * H, H, qkv_v, dev->err);
  g.seq = seq;
  g.qp = mb(qp);
  g.kp = mb(kp);
  g.wq = cb(q_norm_w);
  g.wk = cb(k_norm_w);
  g.rope_cos = rope_cos;
  g.rope_sin = rope_sin;
  g.rope_bstride = rope_bstride;
  g.hidden = H;
  g.heads = n_heads;
  g.eps = eps;
  return run_gemm(dev, mi::EPI_QKV_ROPE, ta, tb, g, static_cast<cudaStream_t>(stream));
}

mi_status mi_qk_norm_rope(const void* qkv, const void* q_norm_w, const void* k_norm_w, const float* rope_cos,
                          const float* rope_sin, int rope_bstride, void* qp, void* kp, int batch, int seq, int n_heads,
                          float eps, void* stream) {
  if (!qkv || !q_norm_w || !k_norm_w || !rope_cos || !rope_sin || !qp || !kp)
    return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(qkv) || !aligned16(q_norm_w) || !aligned16(k_norm_w) || !aligned16(rope_cos) || !aligned16(rope_sin) ||
      !aligned16(qp) || !aligned16(kp))
    return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (batch <= 0 || seq <= 0 || n_heads <= 0) return fail(MI_ERR_INVALID_ARG, "batch, seq, n_heads must be positive");
  if (rope_bstride < 0 || rope_bstride % 4 != 0) return fail(MI_ERR_INVALID_ARG, "bad rope_bstride");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaError_t e = mi::qk_norm_rope_launch(cb(qkv), cb(q_norm_w), cb(k_norm_w), rope_cos, rope_sin, rope_bstride,
                                          mb(qp), mb(kp), batch, seq, n_heads, eps, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "qk_norm_rope");
}

static mi_status attention_common(const void* qp, const void* kp, const void* qkv, const uint8_t* key_mask, void* o,
                                  int batch, int seq, int n_heads, void* ws, size_t ws_bytes, bool use_ws, void* stream) {
  if (!qp || !kp || !qkv || !o) return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(qp) || !aligned16(kp) || !aligned16(qkv) || !aligned16(o))
    return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (batch <= 0 || seq <= 0 || n_heads <= 0) return fail(MI_ERR_INVALID_ARG, "batch, seq, n_heads must be positive");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  const size_t need = use_ws ? mi::attention_scratch_bytes(batch, seq, n_heads, dev->num_sms) : 0;
  if (need > 0) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
      return fail(MI_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
    if (ws_bytes < need) return fail(MI_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, need);
  }
  const int H = n_heads * 128;
  CUtensorMap tq, tk, tv;
  if (!mi::encode_3d_bf16(&tq, qp, 128, (uint64_t)seq, (uint64_t)batch * n_heads, 256, (uint64_t)seq * 256, 64, 128, 1) ||
      !mi::encode_3d_bf16(&tk, kp, 128, (uint64_t)seq, (uint64_t)batch * n_heads, 256, (uint64_t)seq * 256, 64, 128, 1))
    return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (q/k)");
  const uint64_t dims[4] = {128, (uint64_t)n_heads, (uint64_t)seq, (uint64_t)batch};
  const uint64_t str[3] = {256, (uint64_t)3 * H * 2, (uint64_t)seq * 3 * H * 2};
  const uint32_t box[4] = {64, 1, 128, 1};
  if (!mi::encode_4d_bf16(&tv, cb(qkv) + 2 * H, dims, str, box)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (v)");
  mi::AttnArgs aa;
  aa.batch = batch;
  aa.seq = seq;
  aa.n_heads = n_heads;
  aa.key_mask = key_mask;
  aa.out = mb(o);
  aa.scale_log2 = 1.4426950408889634f / sqrtf(128.0f);
  aa.err = dev->err;
  aa.part = nullptr;
  aa.count = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (need > 0) {
    const size_t cb_bytes = mi::attention_count_bytes(batch, seq, n_heads);
    aa.count = static_cast<int*>(ws);
    aa.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + cb_bytes);
    cudaError_t e = cudaMemsetAsync(aa.count, 0, cb_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "attention counters");
  }
  cudaError_t e = mi::attention_launch(tq, tk, tv, aa, dev->num_sms, s);
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "attention launch");
}

mi_status mi_attention(const void* qp, const void* kp, const void* qkv, const uint8_t* key_mask, void* o, int batch,
                       int seq, int n_heads, void* stream) {
  return attention_common(qp, kp, qkv, key_mask, o, batch, seq, n_heads, nullptr, 0, false, stream);
}

mi_status mi_attention_workspace_size(int batch, int seq, int n_heads, size_t* bytes) {
  if (!bytes) return fail(MI_ERR_INVALID_ARG, "null output pointer");
  if (batch <= 0 || seq <= 0 || n_heads <= 0) return fail(MI_ERR_INVALID_ARG, "batch, seq, n_heads must be positive");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  *bytes = mi::attention_scratch_bytes(batch, seq, n_heads, dev->num_sms);
  return MI_OK;
}

mi_status mi_attention_ws(const void* qp, const void* kp, const void* qkv, const uint8_t* key_mask, void* o, int batch,
                          int seq, int n_heads, void* ws, size_t ws_bytes, void* stream) {
  return attention_common(qp, kp, qkv, key_mask, o, batch, seq, n_heads, ws, ws_bytes, true, stream);
}

mi_status mi_gated_add(const void* x, const void* y, const void* mod, int gate_row, void* out, int batch, int seq,
                       int hidden, void* stream) {
  if (!x || !y || !mod || !out) return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(x) || !aligned16(y) || !aligned16(mod) || !aligned16(out))
    return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (batch <= 0 || seq <= 0 || hidden <= 0 || hidden % 8 != 0) return fail(MI_ERR_INVALID_ARG, "bad shape");
  if (gate_row < 0 || gate_row > 5) return fail(MI_ERR_INVALID_ARG, "gate_row is 0..5");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaError_t e = mi::gated_add_launch(cb(x), cb(y), cb(mod) + (size_t)gate_row * hidden, 6 * hidden, mb(out),
                                       batch * seq, seq, hidden, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "gated_add");
}

mi_status mi_silu_gate(const void* gu, void* m, int rows, int inter, void* stream) {
  if (!gu || !m) return fail(MI_ERR_INVALID_ARG, "null tensor argument");
  if (!aligned16(gu) || !aligned16(m)) return fail(MI_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (rows <= 0 || inter <= 0 || inter % 8 != 0) return fail(MI_ERR_INVALID_ARG, "bad shape");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaError_t e = mi::silu_gate_launch(cb(gu), mb(m), rows, inter, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "silu_gate");
}

}  // extern "C"

// ------------------------------------------------------------------------------ static workspace
// A block forward for callers that cannot allocate device memory themselves.  Its workspace is a
// file-scope device array of fixed size that every GPU loading this library holds until the
// process exits.  Host code must not use the array's name as a device address; the address is
// looked up once per device with cudaGetSymbolAddress, with that device current.
namespace {

constexpr size_t kStaticWsBytes = (size_t)64 << 20;
static_assert(kStaticWsBytes == MI_STATIC_WS_BYTES, "the header states the static workspace size");
__device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

void* g_static_ws_ptr[mi::kMaxDevices] = {};
std::mutex g_static_ws_mu;

mi_status static_ws_address(void** out) {
  int dev = 0;
  MI_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= mi::kMaxDevices) return fail(MI_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_static_ws_mu);
  if (!g_static_ws_ptr[dev]) {
    void* p = nullptr;
    MI_CUDA(cudaGetSymbolAddress(&p, g_static_ws), "cudaGetSymbolAddress(static workspace)");
    g_static_ws_ptr[dev] = p;
  }
  *out = g_static_ws_ptr[dev];
  return MI_OK;
}

}  // namespace

extern "C" mi_status mi_block_forward_static_ws(mi_block* blk, const mi_seq_layout* L, const void* x, void* y,
                                                const void* mod, const float* rope_cos, const float* rope_sin,
                                                int rope_bstride, const uint8_t* key_mask, void* stream) {
  if (!blk) return fail(MI_ERR_INVALID_ARG, "null block");
  int S = 0;
  mi_status st = check_layout(L, &S);
  if (st != MI_OK) return st;
  const size_t need = plan_ws(blk->d, L->batch, S, blk->num_sms).total;
  if (need > kStaticWsBytes)
    return fail(MI_ERR_WORKSPACE, "this geometry needs a %zu-byte workspace; the static one holds %zu bytes", need,
                kStaticWsBytes);
  void* ws = nullptr;
  st = static_ws_address(&ws);
  if (st != MI_OK) return st;
  return mi_block_forward(blk, L, x, y, mod, rope_cos, rope_sin, rope_bstride, key_mask, ws, kStaticWsBytes, stream);
}

// ------------------------------------------------------------------------------ device builders
struct mi_tmod {
  mi_tmod_desc d;
  CUtensorMap tm_w1, tm_w2, tm_wmod;
};

namespace {

constexpr int kTDim = 256;
constexpr double kTScale = 1000.0;
constexpr double kTMaxPeriod = 10000.0;

struct TmodLayout {
  size_t emb, a1, c, all, total;
};

TmodLayout plan_tmod(const mi_tmod_desc& d, int batch) {
  TmodLayout l;
  const size_t H = d.hidden, rows_all = (size_t)(6 * d.n_blocks + 2) * H;
  size_t cur = 0;
  l.emb = cur;
  cur = align_up(cur + (size_t)batch * kTDim * 2, 1024);
  l.a1 = cur;
  cur = align_up(cur + (size_t)batch * H * 2, 1024);
  l.c = cur;
  cur = align_up(cur + (size_t)batch * H * 2, 1024);
  l.all = cur;
  cur = align_up(cur + (size_t)batch * rows_all * 2, 1024);
  l.total = cur;
  return l;
}

}  // namespace

extern "C" {

mi_status mi_tmod_init(mi_tmod** out, const mi_tmod_desc* desc) {
  if (!out || !desc) return fail(MI_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  if (desc->hidden <= 0 || desc->hidden % 256 != 0) return fail(MI_ERR_UNSUPPORTED, "hidden must be a multiple of 256");
  if (desc->n_blocks <= 0) return fail(MI_ERR_INVALID_ARG, "n_blocks must be positive");
  if (!desc->w_t1 || !desc->w_t2 || !desc->w_mod || !aligned16(desc->w_t1) || !aligned16(desc->w_t2) ||
      !aligned16(desc->w_mod))
    return fail(MI_ERR_INVALID_ARG, "weights must be non-null and 16-byte aligned");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  mi_tmod* m = new (std::nothrow) mi_tmod;
  if (!m) return fail(MI_ERR_INVALID_ARG, "host allocation failed");
  m->d = *desc;
  const int H = desc->hidden;
  if (!map_w(&m->tm_w1, desc->w_t1, H, kTDim, kWBox) || !map_w(&m->tm_w2, desc->w_t2, H, H, kWBox) ||
      !map_w(&m->tm_wmod, desc->w_mod, (6 * desc->n_blocks + 2) * H, H, kWBox)) {
    delete m;
    return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed (timestep weights)");
  }
  *out = m;
  return MI_OK;
}

void mi_tmod_destroy(mi_tmod* tm) { delete tm; }

mi_status mi_tmod_workspace_size(const mi_tmod* tm, int batch, size_t* bytes) {
  if (!tm || !bytes || batch <= 0) return fail(MI_ERR_INVALID_ARG, "bad argument");
  *bytes = plan_tmod(tm->d, batch).total;
  return MI_OK;
}

mi_status mi_timestep_modulation(mi_tmod* tm, const float* t, int batch, void* mods, void* mod_final, void* ws,
                                 size_t ws_bytes, void* stream) {
  if (!tm || !t || !mods || !mod_final) return fail(MI_ERR_INVALID_ARG, "null argument");
  if (batch <= 0 || batch > 128) return fail(MI_ERR_INVALID_ARG, "batch must be in [1, 128]");
  if (!aligned16(mods) || !aligned16(mod_final)) return fail(MI_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
  const TmodLayout l = plan_tmod(tm->d, batch);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(MI_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
  if (ws_bytes < l.total) return fail(MI_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, l.total);
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = tm->d.hidden, nb = tm->d.n_blocks;
  uint8_t* base = static_cast<uint8_t*>(ws);
  bf16* emb = mb(base + l.emb);
  bf16* a1 = mb(base + l.a1);
  bf16* c = mb(base + l.c);
  bf16* all = mb(base + l.all);
  cudaError_t e = mi::timestep_embedding_launch(t, emb, batch, kTDim, kTScale, kTMaxPeriod, s);
  if (e != cudaSuccess) return cuda_fail(e, "timestep embedding");
  CUtensorMap ta;
  if (!map_a(&ta, emb, batch, kTDim)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed");
  st = run_gemm(dev, mi::EPI_STORE, ta, tm->tm_w1, gemm_args(batch, H, kTDim, a1, dev->err), s);
  if (st != MI_OK) return st;
  e = mi::silu_inplace_launch(a1, (long long)batch * H, s);
  if (e != cudaSuccess) return cuda_fail(e, "silu");
  if (!map_a(&ta, a1, batch, H)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed");
  st = run_gemm(dev, mi::EPI_STORE, ta, tm->tm_w2, gemm_args(batch, H, H, c, dev->err), s);
  if (st != MI_OK) return st;
  e = mi::silu_inplace_launch(c, (long long)batch * H, s);
  if (e != cudaSuccess) return cuda_fail(e, "silu");
  if (!map_a(&ta, c, batch, H)) return fail(MI_ERR_INVALID_ARG, "tensor map encoding failed");
  st = run_gemm(dev, mi::EPI_STORE, ta, tm->tm_wmod, gemm_args(batch, (6 * nb + 2) * H, H, all, dev->err), s);
  if (st != MI_OK) return st;
  e = mi::modulation_split_launch(all, mb(mods), mb(mod_final), batch, nb, H, s);
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "modulation split");
}

mi_status mi_rope_tables(int text_pad, int grid_h, int grid_w, float theta, float* rope_cos, float* rope_sin,
                         void* stream) {
  if (!rope_cos || !rope_sin) return fail(MI_ERR_INVALID_ARG, "null argument");
  if (text_pad < 0 || grid_h < 0 || grid_w <= 0 || !(theta > 1.0f)) return fail(MI_ERR_INVALID_ARG, "bad geometry");
  const long long S = (long long)text_pad + (long long)grid_h * grid_w;
  if (S <= 0 || S > (1 << 20)) return fail(MI_ERR_INVALID_ARG, "sequence length out of range");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaError_t e = mi::rope_table_launch(rope_cos, rope_sin, (int)S, text_pad, grid_w, (double)theta,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "rope tables");
}

mi_status mi_time_advance(float* t, int n, float dt, void* stream) {
  if (!t || n <= 0) return fail(MI_ERR_INVALID_ARG, "bad argument");
  DeviceInfo* dev = nullptr;
  mi_status st = require_sm103(&dev);
  if (st != MI_OK) return st;
  cudaError_t e = mi::time_advance_launch(t, n, dt, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MI_OK : cuda_fail(e, "time advance");
}

}  // extern "C"
