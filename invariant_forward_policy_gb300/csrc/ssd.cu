// Mamba-2 scan in chunked (state-space duality) form, one arithmetic for
// prefill, chunked prefill and decode.
//
// "vLLM Achieves Bitwise-Consistent RL Training ..." §6 ("Transfer: Nemotron,
// a Mamba hybrid architecture + NVFP4"): Mamba-2 is a linear recurrence, and
// decode replays prefill's chunked arithmetic instead of its own single-step
// recurrence.
//
// Per head: state_t = a_t state_{t-1} + B_t x_t^T, y_t = C_t^T state_t, with
// a_t = exp(loga_t).  Chunks are absolute positions [cQ, cQ + Q).  For the row
// at offset i of chunk c, with H_c the state entering the chunk and
// L_i = loga_0 + ... + loga_i (offsets of the chunk, summed in order):
//     y_i = exp(L_i) (C_i^T H_c) + sum_{j = 0..i} (exp(L_i - L_j) (C_i . B_j)) x_j
// and, once the chunk is complete,
//     H_{c+1} = exp(L_{Q-1}) H_c + sum_{j = 0..Q-1} (exp(L_{Q-1} - L_j) B_j) x_j^T.
// Every dot product and sum runs in ascending index order with one fused
// multiply-add per term.  A call processes one piece (a run of consecutive
// positions) per sequence; a per-sequence store keeps H_c and the inputs of
// the chunk's earlier positions (B, x, loga, copied exactly, per head), so a decode step
// or a prefill chunk that starts mid-chunk computes its rows exactly as a
// prefill over the whole chunk does.
#include <algorithm>
#include <mutex>
#include <string>

#include "common.cuh"

namespace bi {

constexpr int kSsdThreads = 256;
constexpr int kSsdMaxQ = 64, kSsdMaxN = 128, kSsdMaxP = 128;
constexpr int kSsdPrefetch = (2 * kSsdMaxQ * kSsdMaxN / 8 + kSsdMaxQ * kSsdMaxP / 8 + kSsdThreads - 1) / kSsdThreads;

struct SsdArgs {
  const __nv_bfloat16* x;  // [T, H, P]
  const __nv_bfloat16* B;  // [T, G, N]
  const __nv_bfloat16* C;  // [T, G, N]
  const float* loga;       // [T, H]
  const int32_t* seq;      // [pieces]
  const int32_t* row0;     // [pieces + 1]
  const int32_t* pos0;     // [pieces]
  float* store;            // [n_seq, floats per sequence]
  float* y;                // [T, H, P]
  int* status;
  int64_t n_seq, store_floats;
  int H, G, P, N, Q;
};

// Per sequence: entering state [H][N][P], then the open chunk's earlier inputs
// B [Q][H][N], x [Q][H][P], loga [Q][H].  B is kept per head (not per group) so
// that each CTA reads and writes only its own slots.
__host__ __device__ inline int64_t ssd_store_floats(int H, int /*G*/, int P, int N, int Q) {
  return (int64_t)H * N * P + (int64_t)Q * H * N + (int64_t)Q * H * P + (int64_t)Q * H;
}

__global__ void __launch_bounds__(kSsdThreads, 2) ssd_scan_kernel(const SsdArgs a) {
  extern __shared__ __align__(16) float sm[];
  const int Q = a.Q, N = a.N, P = a.P, H = a.H, G = a.G;
  // B, C and x hold bf16 values (inputs, or their exact copies in the store):
  // staged as bf16 and widened exactly on use, so that two CTAs share an SM
  // B and C are kept transposed, [n][offset] with row stride QS: a thread's four
  // offsets at one n are one 8-byte load, and a warp's 16 row blocks hit distinct banks
  const int QS = Q + 4;
  float* Hs = sm;                            // [N][P] state entering the chunk
  const int GS = Q + 1;                      // Gm row stride: rows ib and ib + 4 on different banks
  float* Gm = Hs + N * P;                    // [Q][GS] (C_i . B_j) scaled by the decay
  __nv_bfloat16* Bs = reinterpret_cast<__nv_bfloat16*>(Gm + Q * GS);  // [N][QS]
  __nv_bfloat16* Cs = Bs + N * QS;                                   // [N][QS]
  __nv_bfloat16* xs = Cs + N * QS;                                   // [Q][P]
  float* ls = reinterpret_cast<float*>(xs + Q * P);                  // [Q] loga
  float* Ls = ls + Q;             // [Q] cumulative
  float* eL = Ls + Q;             // [Q] exp(L_i)
  float* dq = eL + Q;             // [Q] exp(L_{Q-1} - L_j), for the exit state
  pdl_trigger();
  pdl_wait();
  const int piece = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int g = h / (H / G);
  const int row0 = a.row0[piece];
  const int n_tok = a.row0[piece + 1] - row0;
  if (n_tok <= 0) return;
  const int s = a.seq[piece];
  const int64_t p0 = a.pos0[piece], p1 = p0 + n_tok;
  if (s < 0 || s >= a.n_seq || p0 < 0) {
    if (tid == 0) report(a.status, DEV_BAD_INDEX);
    return;
  }
  float* st = a.store + (int64_t)s * a.store_floats;
  float* st_H = st + (int64_t)h * N * P;                       // [H][N][P]
  float* st_B = st + (int64_t)H * N * P;                       // [Q][H][N]
  float* st_x = st_B + (int64_t)Q * H * N;                     // [Q][H][P]
  float* st_l = st_x + (int64_t)Q * H * P;                     // [Q][H]

  for (int i = tid; i < N * P; i += kSsdThreads) Hs[i] = st_H[i];
  bool advanced = false;  // some chunk completed in this call: the stored state changes
  const int64_t c_first = p0 / Q, c_last = (p1 - 1) / Q;
  // The next chunk's B, C and x (16-byte vectors: B rows, C rows, x rows) are
  // loaded into registers while the current chunk computes; with N and P
  // multiples of 8 (else every chunk is staged directly).  A warp loads whole
  // rows: that measured faster than 16-row groups, whose transposed stores into
  // shared memory would be conflict-free but whose loads span 16 rows.
  const bool vec = N % 8 == 0 && P % 8 == 0;
  const int vb = Q * N / 8, vx = Q * P / 8;  // vectors of B (and of C), of x
  uint4 pf[kSsdPrefetch];
  auto prefetch = [&](int64_t c) {
    const int64_t cs = c * Q;
    const int i1 = (int)((p1 < cs + Q ? p1 : cs + Q) - cs);  // chunks after the first start at offset 0
#pragma unroll
    for (int k = 0; k < kSsdPrefetch; ++k) {
      const int v = tid + k * kSsdThreads;
      if (v < 2 * vb) {
        const int w = v < vb ? v : v - vb, i = w / (N / 8), j = w % (N / 8);
        if (i < i1) {
          const int64_t r = row0 + (cs + i - p0);
          pf[k] = __ldg(reinterpret_cast<const uint4*>((v < vb ? a.B : a.C) + (r * G + g) * N) + j);
        }
      } else if (v < 2 * vb + vx) {
        const int w = v - 2 * vb, i = w / (P / 8), j = w % (P / 8);
        if (i < i1) {
          const int64_t r = row0 + (cs + i - p0);
          pf[k] = __ldg(reinterpret_cast<const uint4*>(a.x + (r * (int64_t)H + h) * P) + j);
        }
      }
    }
  };
  auto place = [&](int i1) {  // the prefetched vectors into Bs, Cs, xs
#pragma unroll
    for (int k = 0; k < kSsdPrefetch; ++k) {
      const int v = tid + k * kSsdThreads;
      if (v < 2 * vb) {
        const int w = v < vb ? v : v - vb, i = w / (N / 8), j = w % (N / 8);
        if (i < i1) {
          // the vector's 8 values go to 8 rows n of the transposed array; lanes
          // start at different rows (r = (j / 2) mod 8) so that a warp's 2-byte
          // stores of one step fall on distinct banks: rotate the values by r first
          __nv_bfloat16* d = (v < vb ? Bs : Cs) + (j * 8) * QS + i;
          const int r = (j >> 1) & 7;
          uint32_t w0 = pf[k].x, w1 = pf[k].y, w2 = pf[k].z, w3 = pf[k].w, t0;
          if (r & 2) {  // by one word
            t0 = w0; w0 = w1; w1 = w2; w2 = w3; w3 = t0;
          }
          if (r & 4) {  // by two words
            t0 = w0; w0 = w2; w2 = t0;
            t0 = w1; w1 = w3; w3 = t0;
          }
          if (r & 1) {  // by one value
            t0 = w0;
            w0 = __funnelshift_r(w0, w1, 16);
            w1 = __funnelshift_r(w1, w2, 16);
            w2 = __funnelshift_r(w2, w3, 16);
            w3 = __funnelshift_r(w3, t0, 16);
          }
          const uint32_t wd[4] = {w0, w1, w2, w3};
#pragma unroll
          for (int t = 0; t < 8; ++t)  // wd's value t is the vector's value (t + r) mod 8
            d[((t + r) & 7) * QS] = __ushort_as_bfloat16((unsigned short)(wd[t >> 1] >> (16 * (t & 1))));
        }
      } else if (v < 2 * vb + vx) {
        const int w = v - 2 * vb, i = w / (P / 8), j = w % (P / 8);
        if (i < i1) *reinterpret_cast<uint4*>(xs + i * P + j * 8) = pf[k];
      }
    }
  };
  for (int64_t c = c_first; c <= c_last; ++c) {
    const int64_t cs = c * Q;
    const int i0 = (int)((p0 > cs ? p0 : cs) - cs), i1 = (int)((p1 < cs + Q ? p1 : cs + Q) - cs);
    if (vec && c > c_first) {
      place(i1);  // i0 == 0 here
    } else {
    // chunk inputs: earlier offsets from the store (first chunk of the call only), new ones from the call
    for (int e = tid; e < i1 * N; e += kSsdThreads) {
      const int i = e / N, n = e % N;
      if (i < i0) {
        Bs[n * QS + i] = f2bf(st_B[((int64_t)i * H + h) * N + n]);  // a bf16 value: exact
      } else {
        const int64_t r = row0 + (cs + i - p0);
        Bs[n * QS + i] = a.B[(r * G + g) * N + n];
        Cs[n * QS + i] = a.C[(r * G + g) * N + n];
      }
    }
    for (int e = tid; e < i1 * P; e += kSsdThreads) {
      const int i = e / P, p = e % P;
      xs[e] = i < i0 ? f2bf(st_x[((int64_t)i * H + h) * P + p])
                     : a.x[((row0 + (cs + i - p0)) * (int64_t)H + h) * P + p];
    }
    }
    for (int i = tid; i < i1; i += kSsdThreads)
      ls[i] = i < i0 ? st_l[(int64_t)i * H + h] : a.loga[(row0 + (cs + i - p0)) * (int64_t)H + h];
    __syncthreads();
    if (vec && c < c_last) prefetch(c + 1);  // in flight while this chunk computes
    if (tid == 0) {
      float acc = 0.f;
      for (int i = 0; i < i1; ++i) {
        acc = __fadd_rn(acc, ls[i]);
        Ls[i] = acc;
      }
    }
    __syncthreads();
    for (int i = tid; i < i1; i += kSsdThreads) {
      eL[i] = expf(Ls[i]);
      if (i1 == Q) dq[i] = expf(__fsub_rn(Ls[Q - 1], Ls[i]));
    }
    // decay-scaled (C_i . B_j) for the rows this call computes; 4 x 4 tiles of (i, j)
    // (row tiles start at a multiple of 4: rows below i0 are computed and dropped)
    const int ia = i0 & ~3;
    {
      const int ni = (i1 - ia + 3) / 4, nj = (i1 + 3) / 4;
      for (int e = tid; e < ni * nj; e += kSsdThreads) {
        const int ib = ia + (e / nj) * 4, jb = (e % nj) * 4;
        if (jb > ib + 3) continue;  // above the diagonal
        float acc[4][4] = {};
        for (int n = 0; n < N; ++n) {
          const uint2 cw = *reinterpret_cast<const uint2*>(Cs + n * QS + ib);
          const uint2 bw = *reinterpret_cast<const uint2*>(Bs + n * QS + jb);
          const float c[4] = {bf16lo(cw.x), bf16hi(cw.x), bf16lo(cw.y), bf16hi(cw.y)};
          const float bb[4] = {bf16lo(bw.x), bf16hi(bw.x), bf16lo(bw.y), bf16hi(bw.y)};
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = __fmaf_rn(c[u], bb[v], acc[u][v]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int i = ib + u, j = jb + v;
            if (i >= i0 && i < i1 && j <= i) Gm[i * GS + j] = __fmul_rn(expf(__fsub_rn(Ls[i], Ls[j])), acc[u][v]);
          }
      }
    }
    __syncthreads();
    // rows: 4 x 4 tiles of (i, p)
    {
      const int ni = (i1 - ia + 3) / 4, np4 = P / 4;
      for (int e = tid; e < ni * np4; e += kSsdThreads) {
        const int ib = ia + (e / np4) * 4, pb = (e % np4) * 4;
        float inter[4][4] = {}, intra[4][4] = {};
        for (int n = 0; n < N; ++n) {
          const float4 hv = *reinterpret_cast<const float4*>(&Hs[n * P + pb]);
          const float hh[4] = {hv.x, hv.y, hv.z, hv.w};
          const uint2 cw = *reinterpret_cast<const uint2*>(Cs + n * QS + ib);
          const float c4[4] = {bf16lo(cw.x), bf16hi(cw.x), bf16lo(cw.y), bf16hi(cw.y)};
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) inter[u][v] = __fmaf_rn(c4[u], hh[v], inter[u][v]);
        }
        const int jmax = ib + 3 < i1 - 1 ? ib + 3 : i1 - 1;
        for (int j = 0; j <= jmax; ++j) {
          const uint2 xr = *reinterpret_cast<const uint2*>(&xs[j * P + pb]);
          const float xx[4] = {bf16lo(xr.x), bf16hi(xr.x), bf16lo(xr.y), bf16hi(xr.y)};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (j > ib + u) continue;  // row ib+u sums j = 0 .. ib+u only
            const float gm = Gm[(ib + u) * GS + j];
#pragma unroll
            for (int v = 0; v < 4; ++v) intra[u][v] = __fmaf_rn(gm, xx[v], intra[u][v]);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = ib + u;
          if (i < i0 || i >= i1) continue;
          const int64_t r = row0 + (cs + i - p0);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            a.y[(r * H + h) * P + pb + v] = __fadd_rn(__fmul_rn(eL[i], inter[u][v]), intra[u][v]);
        }
      }
    }
    if (i1 == Q) {
      // the chunk is complete: its exit state enters the next chunk; 4 x 4 tiles of (n, p)
      __syncthreads();
      const float eLast = eL[Q - 1];
      const int nn4 = N / 4, np4 = P / 4;
      for (int e = tid; e < nn4 * np4; e += kSsdThreads) {
        const int nb = (e / np4) * 4, pb = (e % np4) * 4;
        float acc[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = __fmul_rn(eLast, Hs[(nb + u) * P + pb + v]);
        for (int j = 0; j < Q; ++j) {
          const uint2 xr = *reinterpret_cast<const uint2*>(&xs[j * P + pb]);
          const float xx[4] = {bf16lo(xr.x), bf16hi(xr.x), bf16lo(xr.y), bf16hi(xr.y)};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float wb = __fmul_rn(dq[j], bf2f(Bs[(nb + u) * QS + j]));
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] = __fmaf_rn(wb, xx[v], acc[u][v]);
          }
        }
        // a thread reads and writes only its own tile of Hs here
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) Hs[(nb + u) * P + pb + v] = acc[u][v];
      }
      advanced = true;
    } else {
      // the chunk stays open: keep the inputs of the new offsets for the calls that finish it
      for (int e = tid; e < (i1 - i0) * P; e += kSsdThreads) {
        const int i = i0 + e / P, p = e % P;
        st_x[((int64_t)i * H + h) * P + p] = bf2f(xs[i * P + p]);
      }
      for (int e = tid; e < (i1 - i0) * N; e += kSsdThreads) {
        const int i = i0 + e / N, n = e % N;
        st_B[((int64_t)i * H + h) * N + n] = bf2f(Bs[n * QS + i]);
      }
      for (int i = i0 + tid; i < i1; i += kSsdThreads) st_l[(int64_t)i * H + h] = ls[i];
    }
    __syncthreads();
  }
  // the state entering the sequence's next position (unchanged unless a chunk completed)
  if (advanced)
    for (int i = tid; i < N * P; i += kSsdThreads) st_H[i] = Hs[i];
}

// Decode steps (one position per piece): the same row and exit-state
// arithmetic as ssd_scan_kernel, term for term and in the same order, with the
// entering state and the chunk's earlier inputs read straight from the store
// instead of staged in shared memory, so that many CTAs share an SM.
__global__ void __launch_bounds__(128, 8) ssd_step_kernel(const SsdArgs a) {
  __shared__ float c_s[kSsdMaxN], gm[kSsdMaxQ], Ls[kSsdMaxQ], dq[kSsdMaxQ], b_s[kSsdMaxN], x_s[kSsdMaxP];
  __shared__ float l_s[kSsdMaxQ];
  pdl_trigger();
  pdl_wait();
  const int Q = a.Q, N = a.N, P = a.P, H = a.H, G = a.G;
  const int piece = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int g = h / (H / G);
  const int row0 = a.row0[piece];
  if (a.row0[piece + 1] - row0 != 1) {  // this kernel takes single-position pieces only
    if (a.row0[piece + 1] - row0 > 1 && tid == 0) report(a.status, DEV_BAD_INDEX);
    return;
  }
  const int s = a.seq[piece];
  const int64_t pos = a.pos0[piece];
  if (s < 0 || s >= a.n_seq || pos < 0) {
    if (tid == 0) report(a.status, DEV_BAD_INDEX);
    return;
  }
  float* st = a.store + (int64_t)s * a.store_floats;
  float* st_H = st + (int64_t)h * N * P;
  float* st_B = st + (int64_t)H * N * P;
  float* st_x = st_B + (int64_t)Q * H * N;
  float* st_l = st_x + (int64_t)Q * H * P;
  const int i = (int)(pos % Q);
  const int64_t r = row0;
  for (int n = tid; n < N; n += 128) {
    c_s[n] = bf2f(a.C[(r * G + g) * N + n]);
    b_s[n] = bf2f(a.B[(r * G + g) * N + n]);
  }
  for (int p = tid; p < P; p += 128) x_s[p] = bf2f(a.x[(r * H + h) * P + p]);
  for (int j = tid; j <= i; j += 128) l_s[j] = j < i ? st_l[(int64_t)j * H + h] : a.loga[r * H + h];
  __syncthreads();
  if (tid == 0) {
    float acc = 0.f;
    for (int j = 0; j <= i; ++j) {
      acc = __fadd_rn(acc, l_s[j]);
      Ls[j] = acc;
    }
  }
  __syncthreads();
  for (int j = tid; j <= i; j += 128) {
    const float* bj = j < i ? st_B + ((int64_t)j * H + h) * N : b_s;
    float d = 0.f;
    for (int n = 0; n < N; ++n) d = __fmaf_rn(c_s[n], bj[n], d);
    gm[j] = __fmul_rn(expf(__fsub_rn(Ls[i], Ls[j])), d);
    if (i == Q - 1) dq[j] = expf(__fsub_rn(Ls[Q - 1], Ls[j]));
  }
  __syncthreads();
  const float eLi = expf(Ls[i]);
  for (int p = tid; p < P; p += 128) {
    float inter = 0.f;
    for (int n = 0; n < N; ++n) inter = __fmaf_rn(c_s[n], st_H[(int64_t)n * P + p], inter);
    float intra = 0.f;
    for (int j = 0; j <= i; ++j)
      intra = __fmaf_rn(gm[j], j < i ? st_x[((int64_t)j * H + h) * P + p] : x_s[p], intra);
    a.y[(r * H + h) * P + p] = __fadd_rn(__fmul_rn(eLi, inter), intra);
  }
  if (i == Q - 1) {
    // the position completes its chunk: the exit state replaces the stored one
    __syncthreads();  // every thread has read st_H for its row
    // 4 x 4 tiles of (n, p), each element's terms in ascending j as in the scan
    // kernel; a tile reads 4 B and 4 x values per j as two 16-byte loads
    const float eLast = eLi;
    const int nn4 = N / 4, np4 = P / 4;
    for (int e = tid; e < nn4 * np4; e += 128) {
      const int nb = (e / np4) * 4, pb = (e % np4) * 4;
      float acc[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = __fmul_rn(eLast, st_H[(nb + u) * P + pb + v]);
      for (int j = 0; j < Q; ++j) {
        float4 bv, xv;
        if (j < i) {
          bv = *reinterpret_cast<const float4*>(st_B + ((int64_t)j * H + h) * N + nb);
          xv = *reinterpret_cast<const float4*>(st_x + ((int64_t)j * H + h) * P + pb);
        } else {
          bv = make_float4(b_s[nb], b_s[nb + 1], b_s[nb + 2], b_s[nb + 3]);
          xv = make_float4(x_s[pb], x_s[pb + 1], x_s[pb + 2], x_s[pb + 3]);
        }
        const float bb[4] = {bv.x, bv.y, bv.z, bv.w}, xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float wb = __fmul_rn(dq[j], bb[u]);
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = __fmaf_rn(wb, xx[v], acc[u][v]);
        }
      }
      // each element is read and written by its own thread only
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) st_H[(nb + u) * P + pb + v] = acc[u][v];
    }
  } else {
    for (int n = tid; n < N; n += 128) st_B[((int64_t)i * H + h) * N + n] = b_s[n];
    for (int p = tid; p < P; p += 128) st_x[((int64_t)i * H + h) * P + p] = x_s[p];
    if (tid == 0) st_l[(int64_t)i * H + h] = l_s[i];
  }
}

}  // namespace bi

extern "C" {

size_t bi_ssd_state_bytes(int H, int G, int P, int N, int Q) {
  if (H <= 0 || G <= 0 || P <= 0 || N <= 0 || Q <= 0 || H % G) return 0;
  return (size_t)bi::ssd_store_floats(H, G, P, N, Q) * sizeof(float);
}

bi_status bi_ssd_chunk_scan(const void* x, const void* B, const void* C, const float* loga, const int32_t* piece_seq,
                            const int32_t* piece_row0, const int32_t* piece_pos0, int64_t pieces, int64_t max_q_len,
                            int H, int G, int P, int N, int Q, void* state, int64_t n_seq, float* y, int mode,
                            void* stream) {
  using namespace bi;
  BI_REQUIRE(pieces >= 0, "bad shape");
  BI_REQUIRE(mode == BI_INVARIANT || mode == BI_FAST, "bad mode");
  if (pieces == 0) return BI_OK;
  BI_REQUIRE(x && B && C && loga && piece_seq && piece_row0 && piece_pos0 && state && y, "null pointer");
  BI_REQUIRE(H > 0 && G > 0 && H % G == 0, "H must be a positive multiple of G");
  BI_REQUIRE(aligned16(state), "state must be 16-byte aligned");
  BI_REQUIRE_SHAPE(Q >= 4 && Q <= kSsdMaxQ && Q % 4 == 0 && N >= 4 && N <= kSsdMaxN && N % 4 == 0 && P >= 4 &&
                       P <= kSsdMaxP && P % 4 == 0,
                   "chunk <= 64, state size <= 128 and head size <= 128, each a multiple of 4");
  BI_REQUIRE(pieces <= 0x7fffffff && H <= 65535 && n_seq > 0 && max_q_len >= 1,
             "bad pieces / heads / sequences / max_q_len");
  // fp32 state, decayed C.B and the per-offset scalars; bf16 B, C (transposed, padded) and x
  auto smem_bytes = [](int q, int n, int p) {
    return (n * p + q * (q + 1) + 4 * q) * 4 + (2 * n * (q + 4) + q * p) * 2;
  };
  const int smem = smem_bytes(Q, N, P);
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    const int mx = smem_bytes(kSsdMaxQ, kSsdMaxN, kSsdMaxP);
    attr_err = cudaFuncSetAttribute(ssd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  });
  if (attr_err != cudaSuccess)
    return fail(BI_ERR_CUDA, std::string("bi_ssd_chunk_scan smem attribute: ") + cudaGetErrorString(attr_err));
  SsdArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.B = static_cast<const __nv_bfloat16*>(B);
  a.C = static_cast<const __nv_bfloat16*>(C);
  a.loga = loga;
  a.seq = piece_seq;
  a.row0 = piece_row0;
  a.pos0 = piece_pos0;
  a.store = static_cast<float*>(state);
  a.y = y;
  a.status = device_status_ptr();
  a.n_seq = n_seq;
  a.store_floats = ssd_store_floats(H, G, P, N, Q);
  a.H = H;
  a.G = G;
  a.P = P;
  a.N = N;
  a.Q = Q;
  // single-position pieces (decode steps) take the lighter schedule: same arithmetic
  if (max_q_len == 1)
    return launched(launch_pdl(ssd_step_kernel, dim3((unsigned)pieces, (unsigned)H), dim3(128), 0, as_stream(stream),
                               a),
                    "bi_ssd_chunk_scan");
  return launched(launch_pdl(ssd_scan_kernel, dim3((unsigned)pieces, (unsigned)H), dim3(kSsdThreads), smem,
                             as_stream(stream), a),
                  "bi_ssd_chunk_scan");
}

}  // extern "C"
