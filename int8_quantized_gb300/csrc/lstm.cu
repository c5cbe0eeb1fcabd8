// lstm.cu -- DynamicQuantizeLSTM (ONNX Runtime contrib schema
// "DynamicQuantizeLSTM"; graiphic.io "DynamicQuantizeLSTM") on the dynamic
// quantized GEMM engine.
//
// int8 W [D, input, 4H] and R [D, H, 4H] with per-channel (or per-direction)
// scales and zero point 0; fp32 X; default activations (sigmoid for the
// i, o, f gates, tanh for the cell candidate and the output); gate column
// order i, o, f, c.  X and each step's hidden state are quantized per row to
// uint8 exactly like A of the dynamic quantized inner product.
//   input projection (all steps at once, both directions): Gx = X W[d]
//   per step t: Gh = h_{t-1} R[d]; g = ((Gx_t + Gh) + Wb) + Rb
//               i, o, f = sigmoid(g); ct = tanh(g_c)
//               c = f*c_{t-1} + i*ct;  h = o*tanh(c)
// The reverse direction walks t = T-1 .. 0.  X is quantized once and shared
// by both directions.
#include "common.cuh"

namespace i8q {
namespace {

struct LstmLayout {
  int64_t D, TB, Ip, Hp, H4;
  size_t off_Wt, off_Wcs, off_Rt, off_Rcs, off_Wsc, off_Rsc, off_uX, off_sX, off_zX, off_Gx, off_uh, off_sh, off_zh,
      off_Gh, off_h, off_c, total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

LstmLayout lstm_layout(int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction) {
  LstmLayout L;
  L.D = direction == I8Q_LSTM_BIDIRECTIONAL ? 2 : 1;
  L.TB = T * batch;
  L.Ip = round_up(input, 64);
  L.Hp = round_up(hidden, 64);
  L.H4 = 4 * hidden;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.off_Wt = take((size_t)L.D * L.H4 * L.Ip);
  L.off_Wcs = take((size_t)L.D * L.H4 * 4);
  L.off_Rt = take((size_t)L.D * L.H4 * L.Hp);
  L.off_Rcs = take((size_t)L.D * L.H4 * 4);
  L.off_Wsc = take((size_t)L.D * L.H4 * 4);
  L.off_Rsc = take((size_t)L.D * L.H4 * 4);
  L.off_uX = take((size_t)L.TB * L.Ip);
  L.off_sX = take((size_t)L.TB * 4);
  L.off_zX = take((size_t)L.TB * 4);
  L.off_Gx = take((size_t)L.D * L.TB * L.H4 * 4);
  L.off_uh = take((size_t)L.D * batch * L.Hp);
  L.off_sh = take((size_t)L.D * batch * 4);
  L.off_zh = take((size_t)L.D * batch * 4);
  L.off_Gh = take((size_t)L.D * batch * L.H4 * 4);
  L.off_h = take((size_t)L.D * 2 * batch * hidden * 4);
  L.off_c = take((size_t)L.D * batch * hidden * 4);
  L.total = o;
  return L;
}

// Expand per-direction scales (n == D) or copy per-channel scales (n == D*4H).
__global__ void expand_scales(const float* __restrict__ src, int64_t n, int64_t D, int64_t H4, float* __restrict__ dst) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < D * H4; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = n == D ? src[i / H4] : src[i];
}

__global__ void init_state(const float* __restrict__ h0, const float* __restrict__ c0, int64_t n, float* __restrict__ h,
                           float* __restrict__ c) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    h[i] = h0 ? h0[i] : 0.0f;
    c[i] = c0 ? c0[i] : 0.0f;
  }
}

__device__ __forceinline__ float sigmoid_f32(float x) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x))); }

// One cell update for one direction: batch x H elements.  c_prev and c_out
// may be the same buffer (each element is read, then written, by one thread).
__global__ void lstm_cell_kernel(const float* __restrict__ Gx, const float* __restrict__ Gh,
                                 const float* __restrict__ Wb, const float* __restrict__ Rb,
                                 const float* c_prev, float* __restrict__ h_out, float* c_out,
                                 float* __restrict__ Y, int64_t batch, int64_t H) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < batch * H; e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = e / H, u = e % H;
    float g[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t n = q * H + u;
      float v = __fadd_rn(Gx[b * 4 * H + n], Gh[b * 4 * H + n]);
      if (Wb) v = __fadd_rn(v, Wb[n]);
      if (Rb) v = __fadd_rn(v, Rb[n]);
      g[q] = v;
    }
    const float ig = sigmoid_f32(g[0]);
    const float og = sigmoid_f32(g[1]);
    const float fg = sigmoid_f32(g[2]);
    const float ct = tanhf(g[3]);
    const float c = __fadd_rn(__fmul_rn(fg, c_prev[e]), __fmul_rn(ig, ct));
    const float h = __fmul_rn(og, tanhf(c));
    c_out[e] = c;
    h_out[e] = h;
    if (Y) Y[e] = h;
  }
}

__global__ void copy_f32(const float* __restrict__ src, float* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

__global__ void any_nonzero_s8(const int8_t* __restrict__ p, int64_t n, int* __restrict__ flag) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    if (p[i] != 0) atomicOr(flag, 1);
}

int grid_for(int64_t n, int threads = 256) {
  return (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, threads), (int64_t)sm_count() * 8));
}

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" size_t i8q_dq_lstm_workspace_size(int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction) {
  if (T <= 0 || batch <= 0 || input <= 0 || hidden <= 0) return 0;
  if (direction < I8Q_LSTM_FORWARD || direction > I8Q_LSTM_BIDIRECTIONAL) return 0;
  return lstm_layout(T, batch, input, hidden, direction).total;
}

extern "C" int i8q_dq_lstm_forward(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden,
                                   int direction, const int8_t* W, const float* W_scale, const int8_t* W_zero_point,
                                   size_t n_wscale, const int8_t* R, const float* R_scale,
                                   const int8_t* R_zero_point, size_t n_rscale, const float* Bias, const float* h0,
                                   const float* c0, float* Y, float* Y_h, float* Y_c, void* workspace,
                                   size_t ws_bytes, void* stream) {
  if (T <= 0 || batch <= 0 || input <= 0 || hidden <= 0)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: T, batch, input, hidden must be positive");
  if (direction < I8Q_LSTM_FORWARD || direction > I8Q_LSTM_BIDIRECTIONAL)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: bad direction");
  if (!X || !W || !R || !W_scale || !R_scale) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: NULL tensor pointer");
  if (input > 65536 || hidden > 65536) return fail(I8Q_ERR_UNSUPPORTED, "dq_lstm: input/hidden > 65536");
  const LstmLayout L = lstm_layout(T, batch, input, hidden, direction);
  if ((int64_t)n_wscale != L.D && (int64_t)n_wscale != L.D * L.H4)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: W_scale must have D or D*4H entries");
  if ((int64_t)n_rscale != L.D && (int64_t)n_rscale != L.D * L.H4)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: R_scale must have D or D*4H entries");
  if (!workspace || ws_bytes < L.total) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: workspace missing or too small");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: workspace not 256-byte aligned");
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int8_t* Wt = (int8_t*)(ws + L.off_Wt);
  int32_t* Wcs = (int32_t*)(ws + L.off_Wcs);
  int8_t* Rt = (int8_t*)(ws + L.off_Rt);
  int32_t* Rcs = (int32_t*)(ws + L.off_Rcs);
  float* Wsc = (float*)(ws + L.off_Wsc);
  float* Rsc = (float*)(ws + L.off_Rsc);
  uint8_t* uX = ws + L.off_uX;
  float* sX = (float*)(ws + L.off_sX);
  int32_t* zX = (int32_t*)(ws + L.off_zX);
  float* Gx = (float*)(ws + L.off_Gx);
  uint8_t* uh = ws + L.off_uh;
  float* sh = (float*)(ws + L.off_sh);
  int32_t* zh = (int32_t*)(ws + L.off_zh);
  float* Gh = (float*)(ws + L.off_Gh);
  float* hbuf = (float*)(ws + L.off_h);
  float* cbuf = (float*)(ws + L.off_c);
  const int64_t H = hidden, BH = batch * hidden;

  // Zero points must be zero (the only form this engine runs).  Checked on
  // the device, reported synchronously.
  if (W_zero_point || R_zero_point) {
    int* flag = reinterpret_cast<int*>(Gh);  // scratch word, overwritten later
    I8Q_CUDA_TRY(cudaMemsetAsync(flag, 0, sizeof(int), s));
    if (W_zero_point) any_nonzero_s8<<<grid_for((int64_t)n_wscale), 256, 0, s>>>(W_zero_point, (int64_t)n_wscale, flag);
    if (R_zero_point) any_nonzero_s8<<<grid_for((int64_t)n_rscale), 256, 0, s>>>(R_zero_point, (int64_t)n_rscale, flag);
    int hflag = 0;
    I8Q_CUDA_TRY(cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, s));
    I8Q_CUDA_TRY(cudaStreamSynchronize(s));
    if (hflag) return fail(I8Q_ERR_UNSUPPORTED, "dq_lstm: nonzero W/R zero points are not supported");
  }

  int rc;
  for (int64_t d = 0; d < L.D; ++d) {
    rc = launch_repack_cols_s8(W + d * input * L.H4, input, L.H4, L.H4, Wt + d * L.H4 * L.Ip, nullptr, L.Ip,
                               Wcs + d * L.H4, s);
    if (rc) return rc;
    rc = launch_repack_cols_s8(R + d * H * L.H4, H, L.H4, L.H4, Rt + d * L.H4 * L.Hp, nullptr, L.Hp, Rcs + d * L.H4, s);
    if (rc) return rc;
  }
  expand_scales<<<grid_for(L.D * L.H4), 256, 0, s>>>(W_scale, (int64_t)n_wscale, L.D, L.H4, Wsc);
  expand_scales<<<grid_for(L.D * L.H4), 256, 0, s>>>(R_scale, (int64_t)n_rscale, L.D, L.H4, Rsc);
  I8Q_LAUNCH_CHECK("expand_scales");

  // input projection: X quantized once, one GEMM per direction
  rc = launch_quantize_rows(X, I8Q_F32, L.TB, input, input, uX, nullptr, L.Ip, sX, zX, s);
  if (rc) return rc;
  for (int64_t d = 0; d < L.D; ++d) {
    GemmEpilogue ep{zX, sX, Wcs + d * L.H4, Wsc + d * L.H4, nullptr, I8Q_ACT_IDENTITY, OUT_F32,
                    Gx + d * L.TB * L.H4, L.H4};
    rc = launch_gemm_imma(uX, Wt + d * L.H4 * L.Ip, L.TB, L.H4, L.Ip, ep, s);
    if (rc) return rc;
  }

  for (int64_t d = 0; d < L.D; ++d)
    init_state<<<grid_for(BH), 256, 0, s>>>(h0 ? h0 + d * BH : nullptr, c0 ? c0 + d * BH : nullptr, BH,
                                             hbuf + d * 2 * BH, cbuf + d * BH);
  I8Q_LAUNCH_CHECK("init_state");

  for (int64_t step = 0; step < T; ++step) {
    for (int64_t d = 0; d < L.D; ++d) {
      const bool rev = direction == I8Q_LSTM_REVERSE || (direction == I8Q_LSTM_BIDIRECTIONAL && d == 1);
      const int64_t t = rev ? T - 1 - step : step;
      float* h_prev = hbuf + d * 2 * BH + (step & 1) * BH;
      float* h_next = hbuf + d * 2 * BH + ((step + 1) & 1) * BH;
      rc = launch_quantize_rows(h_prev, I8Q_F32, batch, H, H, uh + d * batch * L.Hp, nullptr, L.Hp, sh + d * batch,
                                zh + d * batch, s);
      if (rc) return rc;
      GemmEpilogue ep{zh + d * batch, sh + d * batch, Rcs + d * L.H4, Rsc + d * L.H4, nullptr, I8Q_ACT_IDENTITY,
                      OUT_F32, Gh + d * batch * L.H4, L.H4};
      rc = launch_gemm_imma(uh + d * batch * L.Hp, Rt + d * L.H4 * L.Hp, batch, L.H4, L.Hp, ep, s);
      if (rc) return rc;
      const float* Wb = Bias ? Bias + d * 8 * H : nullptr;
      const float* Rb = Bias ? Bias + d * 8 * H + 4 * H : nullptr;
      float* Yt = Y ? Y + (t * L.D + d) * BH : nullptr;
      I8Q_PROF("lstm_cell", s);
      lstm_cell_kernel<<<grid_for(BH), 256, 0, s>>>(Gx + d * L.TB * L.H4 + t * batch * L.H4, Gh + d * batch * L.H4, Wb,
                                                    Rb, cbuf + d * BH, h_next, cbuf + d * BH, Yt, batch, H);
      I8Q_LAUNCH_CHECK("lstm_cell_kernel");
    }
  }
  for (int64_t d = 0; d < L.D; ++d) {
    const float* h_last = hbuf + d * 2 * BH + (T & 1) * BH;
    if (Y_h) copy_f32<<<grid_for(BH), 256, 0, s>>>(h_last, Y_h + d * BH, BH);
    if (Y_c) copy_f32<<<grid_for(BH), 256, 0, s>>>(cbuf + d * BH, Y_c + d * BH, BH);
  }
  I8Q_LAUNCH_CHECK("copy_f32");
  return I8Q_OK;
}
