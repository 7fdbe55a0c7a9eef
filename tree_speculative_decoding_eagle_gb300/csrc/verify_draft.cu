// Stage 4 with draft distributions: speculative-sampling verification of a
// tree whose tokens were drawn from the draft's distribution q.
//
// [EAGLE-1] section "検証方法": a drafted token is accepted by the ratio of the
// target and draft probabilities, min(1, p(t)/q(t)); after a rejection the
// target distribution is replaced by the residual norm(max(0, p - q)) and a
// token is finally drawn from it, so the output follows the target exactly.
// Tree form: at node cur the children (node order, all drafted from q =
// softmax(draft row of cur / T)) are tested in turn against the current
// residual R = max(0, p - C q) with normaliser S (C = 0, S = 1 before any
// rejection; each rejection adds S to C and recomputes S over the vocab):
//   child x with token t is accepted iff u[x,0] * S * q(t) < R(t).
// With no child accepted (or at a leaf) the bonus token is drawn from R by
// inverse CDF with u[cur,1].  A residual that sums to 0 falls back to p.
//
// One CTA per sequence: every decision is taken by all threads on
// block-reduced values, so control flow is block-uniform.  Per node: one pass
// over the target and draft rows for the (max, sum) of p and q, one pass per
// rejection for S, and one for the bonus scan; rows stay in L2 across passes.
#include "common.cuh"

namespace eagle {

constexpr int kVDThreads = 512;
constexpr int kBatch = 4;  // vectors per thread whose loads are in flight together

struct DraftVerifyArgs {
  const void *target, *draft;
  int64_t ld_t, ld_d;
  const int32_t *node_tok, *node_parent, *node_row;
  int B, n, D, k, V;
  float inv_t;
  const float *u;
  int32_t *accept_len, *path_nodes, *out_tokens, *status;
};

// Block-wide sum (all threads get it).  s_red holds one float per warp.
__device__ __forceinline__ float block_sum(float v, float *s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = lane < nw ? s_red[lane] : 0.f;
  return warp_sum(t);
}

// Block-wide (max, sum of exp relative to max) merge of per-thread pairs.
__device__ __forceinline__ void block_lse(float &m, float &s, float *s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2);
  }
  __syncthreads();
  if (lane == 0) {
    s_red[2 * warp] = m;
    s_red[2 * warp + 1] = s;
  }
  __syncthreads();
  m = lane < nw ? s_red[2 * lane] : -INFINITY;
  s = lane < nw ? s_red[2 * lane + 1] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2);
  }
}

template <typename T>
__global__ void __launch_bounds__(kVDThreads) verify_draft_kernel(DraftVerifyArgs a) {
  using VT = VecTraits<T>;
  constexpr int VEC = VT::kElems;
  extern __shared__ __align__(16) int s_nodes[];
  int *s_par = s_nodes, *s_tok = s_nodes + a.n;
  __shared__ float s_red[64];
  __shared__ int s_kids[64 + 1];  // children of the current node (node order), count last
  __shared__ int s_pick;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int n = a.n, V = a.V, nvec = V / VEC;
  const float L2E = kLog2e;
  const float sc = a.inv_t * L2E;  // logit -> base-2 exponent units

  for (int i = tid; i < n; i += blockDim.x) {
    s_par[i] = a.node_parent[static_cast<int64_t>(b) * n + i];
    s_tok[i] = a.node_tok[static_cast<int64_t>(b) * n + i];
  }
  __syncthreads();

  int cur = 0, acc = 0, bonus = -1;
  bool bad = false;
  for (int depth = 0;; ++depth) {
    // children of cur in node order (warp 0, ballot compaction)
    if (tid < 32) {
      int cnt = 0;
      for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const bool kid = i > 0 && i < n && s_par[i] == cur;
        const unsigned bal = __ballot_sync(0xffffffffu, kid);
        const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
        if (kid && pos < 64) s_kids[pos] = i;
        cnt += __popc(bal);
      }
      if (lane == 0) s_kids[64] = min(cnt, 64);
    }
    __syncthreads();
    const int nk = s_kids[64];
    const T *prow = reinterpret_cast<const T *>(a.target) + (static_cast<int64_t>(b) * n + cur) * a.ld_t;
    const T *qrow = nullptr;
    if (nk > 0) {
      const int r = a.node_row[static_cast<int64_t>(b) * n + cur];
      if (r < 0 || r >= a.D * a.k || depth >= a.D) {  // a parent must have been expanded
        bad = true;
        break;
      }
      qrow = reinterpret_cast<const T *>(a.draft) + (static_cast<int64_t>(b) * a.D * a.k + r) * a.ld_d;
    }
    // (max, sum) of p and q in base-2 units: y = x * inv_t * log2(e); each
    // thread's vectors of a batch are loaded before any is used, so a pass
    // costs one memory latency per batch, not one per vector
    float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
    for (int base = 0; base < nvec; base += kBatch * kVDThreads) {
      uint4 bp[kBatch], bq[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int vi = base + k * kVDThreads + tid;
        if (vi < nvec) {
          bp[k] = *reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(vi) * VEC);
          if (qrow) bq[k] = *reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(vi) * VEC);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
      if (base + k * kVDThreads + tid >= nvec) continue;
      float x[VEC];
      VT::unpack(bp[k], x);
      float vm = x[0];
#pragma unroll
      for (int e = 1; e < VEC; ++e) vm = fmaxf(vm, x[e]);
      vm *= sc;
      if (vm > -INFINITY) {  // a vector of -inf logits adds nothing
        const float mn = fmaxf(mp, vm);
        float acc_s = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc_s += ex2_approx(fmaf(x[e], sc, -mn));
        sp = (mp == -INFINITY ? 0.f : sp * ex2_approx(mp - mn)) + acc_s;
        mp = mn;
      }
      if (qrow) {
        VT::unpack(bq[k], x);
        float wm = x[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) wm = fmaxf(wm, x[e]);
        wm *= sc;
        if (wm > -INFINITY) {
          const float mq2 = fmaxf(mq, wm);
          float acc_q = 0.f;
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc_q += ex2_approx(fmaf(x[e], sc, -mq2));
          sq = (mq == -INFINITY ? 0.f : sq * ex2_approx(mq - mq2)) + acc_q;
          mq = mq2;
        }
      }
      }
    }
    // lse_combine works in natural units: convert, merge, convert back
    {
      float m_n = mp * kLn2, s_n = sp;
      block_lse(m_n, s_n, s_red);
      mp = m_n * L2E;
      sp = s_n;
      if (qrow) {
        m_n = mq * kLn2;
        s_n = sq;
        block_lse(m_n, s_n, s_red);
        mq = m_n * L2E;
        sq = s_n;
      }
    }
    const float ip = 1.f / sp, iq = qrow ? 1.f / sq : 0.f;
    // residual R(v) = max(0, p(v) - C q(v)), normaliser S
    float C = 0.f, S = 1.f;
    int accepted = -1;
    for (int c = 0; c < nk; ++c) {
      const int x = s_kids[c];
      const int t = s_tok[x];
      if (t < 0 || t >= V) {
        bad = true;
        break;
      }
      const float pt = ex2_approx(fmaf(VT::load1(prow, t), sc, -mp)) * ip;
      const float qt = ex2_approx(fmaf(VT::load1(qrow, t), sc, -mq)) * iq;
      const float ux = a.u[(static_cast<int64_t>(b) * n + x) * 2];
      if (ux * S * qt < fmaxf(0.f, pt - C * qt)) {
        accepted = x;
        break;
      }
      C += S;
      float part = 0.f;
      for (int base = 0; base < nvec; base += kBatch * kVDThreads) {
        uint4 bp[kBatch], bq[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int vi = base + k * kVDThreads + tid;
          if (vi < nvec) {
            bp[k] = *reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(vi) * VEC);
            bq[k] = *reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(vi) * VEC);
          }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (base + k * kVDThreads + tid >= nvec) continue;
          float xp[VEC], xq[VEC];
          VT::unpack(bp[k], xp);
          VT::unpack(bq[k], xq);
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            part += fmaxf(0.f, ex2_approx(fmaf(xp[e], sc, -mp)) * ip - C * ex2_approx(fmaf(xq[e], sc, -mq)) * iq);
        }
      }
      S = block_sum(part, s_red);
      if (!(S > 0.f)) {  // nothing left: fall back to p
        C = 0.f;
        S = 1.f;
      }
    }
    if (bad) break;
    if (accepted >= 0) {
      if (tid == 0) {
        a.path_nodes[static_cast<int64_t>(b) * (a.D + 1) + acc + 1] = accepted;
        a.out_tokens[static_cast<int64_t>(b) * (a.D + 1) + acc] = s_tok[accepted];
      }
      cur = accepted;
      ++acc;
      continue;
    }
    // bonus: inverse CDF of R; thread t owns a contiguous range of vectors
    const int per = (nvec + blockDim.x - 1) / blockDim.x;
    const int v0 = min(nvec, tid * per), v1 = min(nvec, v0 + per);
    float own = 0.f;
    const bool use_q = qrow && C > 0.f;
    for (int vb = v0; vb < v1; vb += kBatch) {
      uint4 bp[kBatch], bq[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (vb + k < v1) {
          bp[k] = *reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(vb + k) * VEC);
          if (use_q) bq[k] = *reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(vb + k) * VEC);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (vb + k >= v1) continue;
        float xp[VEC], xq[VEC];
        VT::unpack(bp[k], xp);
        if (use_q) VT::unpack(bq[k], xq);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float p = ex2_approx(fmaf(xp[e], sc, -mp)) * ip;
          own += use_q ? fmaxf(0.f, p - C * ex2_approx(fmaf(xq[e], sc, -mq)) * iq) : p;
        }
      }
    }
    // exclusive block scan of `own`
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) s_red[tid >> 5] = incl;
    if (tid == 0) s_pick = -1;
    __syncthreads();
    float wbase = 0.f, total = 0.f;
    for (int w = 0; w < (blockDim.x >> 5); ++w) {
      const float ws = s_red[w];
      if (w < (tid >> 5)) wbase += ws;
      total += ws;
    }
    const float before = wbase + incl - own;
    const float thr = a.u[(static_cast<int64_t>(b) * n + cur) * 2 + 1] * total;
    if (own > 0.f && thr >= before && thr < before + own) {
      float run = before;
      int pick = -1;
      for (int vi = v0; vi < v1 && pick < 0; ++vi) {
        float xp[VEC], xq[VEC];
        VT::unpack(*reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(vi) * VEC), xp);
        if (qrow && C > 0.f) VT::unpack(*reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(vi) * VEC), xq);
        for (int e = 0; e < VEC; ++e) {
          const float p = ex2_approx(fmaf(xp[e], sc, -mp)) * ip;
          const float r = (qrow && C > 0.f) ? fmaxf(0.f, p - C * ex2_approx(fmaf(xq[e], sc, -mq)) * iq) : p;
          run += r;
          if (r > 0.f && run > thr) {
            pick = vi * VEC + e;
            break;
          }
        }
      }
      if (pick < 0) pick = v1 * VEC - 1;  // rounding at the range's end
      atomicMax(&s_pick, pick);
    }
    __syncthreads();
    bonus = s_pick;
    if (bonus < 0) {
      // thr at or beyond the rounded total: the last token with mass
      if (own > 0.f) atomicMax(&s_pick, v1 * VEC - 1);
      __syncthreads();
      bonus = s_pick;
    }
    break;
  }
  if (tid == 0) {
    const int64_t ob = static_cast<int64_t>(b) * (a.D + 1);
    a.accept_len[b] = acc;
    a.path_nodes[ob] = 0;
    for (int i = acc + 1; i <= a.D; ++i) a.path_nodes[ob + i] = -1;
    a.out_tokens[ob + acc] = bad ? -1 : bonus;
    for (int i = acc + 1; i <= a.D; ++i) a.out_tokens[ob + i] = -1;
    if (bad || bonus < 0) report(a.status, EAGLE_ERR_INVALID);
  }
}

cudaError_t launch_verify_draft(const void *target, const void *draft, int dtype, int64_t ld_t, int64_t ld_d,
                                const int32_t *node_tok, const int32_t *node_parent, const int32_t *node_row,
                                int B, int m, int D, int k, int V, float temperature, const float *uniforms,
                                int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                                cudaStream_t st) {
  DraftVerifyArgs a;
  a.target = target; a.draft = draft; a.ld_t = ld_t; a.ld_d = ld_d;
  a.node_tok = node_tok; a.node_parent = node_parent; a.node_row = node_row;
  a.B = B; a.n = m + 1; a.D = D; a.k = k; a.V = V;
  a.inv_t = 1.f / temperature;
  a.u = uniforms;
  a.accept_len = accept_len; a.path_nodes = path_nodes; a.out_tokens = out_tokens; a.status = status;
  const size_t smem = sizeof(int) * 2 * static_cast<size_t>(a.n);
  if (dtype == EAGLE_BF16)
    verify_draft_kernel<__nv_bfloat16><<<B, kVDThreads, smem, st>>>(a);
  else
    verify_draft_kernel<float><<<B, kVDThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace eagle
