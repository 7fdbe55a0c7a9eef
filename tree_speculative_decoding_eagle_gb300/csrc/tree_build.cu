// Stage 2: dynamic draft tree (global scores, top-k expansion, top-m
// rerank, node order) and the ancestor-only attention mask.
//
// [EAGLE-2] section "動的ドラフトツリーの構築アルゴリズム": V_i is the product
// of the confidences on the root path; at each depth the k nodes with the
// largest V are expanded, each with its own top-k tokens; the m candidates
// with the largest V are kept and, with their ancestors, form a connected
// tree.  Section "注意マスクの調整": each node attends only to its ancestors.
//
// One CTA per sequence, everything in shared memory.  A candidate is a
// 64-bit key  bits(V):32 | (4095 - parent gid):12 | (2^20 - 1 - token):20,
// so unsigned order is the rank order (V desc, parent gid asc, token asc)
// and keys are unique.  Ranks are obtained by counting larger keys (one
// thread per item, the lanes of a warp reading the same keys).  The running top-m list is merged with each
// new layer by rank arithmetic, so the whole candidate set is never sorted.
//
// Ablation variants ([EAGLE-2] section "実験結果", ablation table), chosen by
// flags: EAGLE_TREE_CONFIDENCE_ONLY ranks a candidate by its own confidence
// c instead of V (expansion and rerank; the rerank then grows the tree
// best-first: the greatest key whose parent is already in the tree, which
// with V keys is the same top-m set); EAGLE_TREE_NO_RERANK keeps the
// layers' selections E_1, E_2, ... (each layer's k best keys) in depth
// order, truncated to m nodes.
#include "common.cuh"

namespace eagle {

constexpr int kTreeThreads = 512;
constexpr int kMaxGid = 4095;

__device__ __forceinline__ uint64_t tree_key(float v, int pgid, int tok) {
  return (static_cast<uint64_t>(__float_as_uint(v)) << 32) |
         (static_cast<uint64_t>(kMaxGid - pgid) << 20) |
         static_cast<uint64_t>(0xFFFFF - tok);
}
__device__ __forceinline__ float tkey_score(uint64_t k) { return __uint_as_float(static_cast<uint32_t>(k >> 32)); }
__device__ __forceinline__ int tkey_parent(uint64_t k) { return kMaxGid - static_cast<int>((k >> 20) & 0xFFF); }
__device__ __forceinline__ int tkey_token(uint64_t k) { return 0xFFFFF - static_cast<int>(k & 0xFFFFF); }

struct TreeArgs {
  const int32_t *tok;
  const float *conf;
  int B, D, k, m, NC, flags;
  const int32_t *root_tok;
  int32_t *node_tok, *node_parent, *node_depth, *node_src, *node_row;
  float *node_score;
  uint64_t *mask;
  int32_t *status;
};

// How many of the n keys of `set` exceed `me`.  Meant for a warp whose
// lanes rank different items against the same set: every load is then a
// shared-memory broadcast, eight in flight.
__device__ __forceinline__ int count_greater(uint64_t me, const uint64_t *set, int n) {
  int c = 0, q = 0;
  for (; q + 8 <= n; q += 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) c += set[q + e] > me;
  }
  for (; q < n; ++q) c += set[q] > me;
  return c;
}

__device__ __forceinline__ int depth_of_gid(int g, int k) {
  if (g == 0) return 0;
  if (g <= k) return 1;
  return 2 + (g - 1 - k) / (k * k);
}
__device__ __forceinline__ int layer_base(int d, int k) {  // first gid of depth d >= 1
  return d == 1 ? 1 : 1 + k + (d - 2) * k * k;
}

// Ancestor-or-self bits of node i, word w, walking parent pointers held in
// shared memory (at most n steps even on malformed input).
__device__ __forceinline__ uint64_t mask_word(const int *par, int n, int i, int w) {
  uint64_t bits = 0;
  int j = i;
  for (int steps = 0; j >= 0 && j < n && steps <= n; ++steps) {
    if ((j >> 6) == w) bits |= 1ull << (j & 63);
    j = par[j];
  }
  return bits;
}

__global__ void __launch_bounds__(kTreeThreads) tree_build_kernel(TreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int k = a.k, m = a.m, NC = a.NC, D = a.D;
  const int kk = k * k;
  const int n = m + 1;
  const int R = 1 + (D - 1) * k;  // used draft rows

  // shared layout
  uint64_t *s_key = reinterpret_cast<uint64_t *>(smem);        // [NC+1] every candidate's key
  uint64_t *s_L = s_key + (NC + 1);                              // [2][m] running top-m keys
  int *s_Lg = reinterpret_cast<int *>(s_L + 2 * m);              // [2][m] their gids
  int *s_cnt = s_Lg + 2 * m;                                     // [2*kk + m] ranks
  int *s_row = s_cnt + (2 * kk + m);                             // [NC+1] gid -> draft row slot
  int *s_out = s_row + (NC + 1);                                 // [NC+1] gid -> output node
  int *s_sel = s_out + (NC + 1);                                 // [m] gids in output order
  int *s_E = s_sel + m;                                          // [k] expanded gids by rank
  int *s_tok = s_E + k;                                          // [R*k] used rows
  float *s_conf = reinterpret_cast<float *>(s_tok + R * k);
  // confidence only: group e's children sorted by key, [R][k] head values
  // (see the pick loop), 8-byte aligned
  uint64_t *s_grec = reinterpret_cast<uint64_t *>((reinterpret_cast<uintptr_t>(s_conf + R * k) + 7) & ~static_cast<uintptr_t>(7));
  __shared__ int s_bad;
  const bool conf_only = (a.flags & EAGLE_TREE_CONFIDENCE_ONLY) != 0;
  const bool rerank = (a.flags & EAGLE_TREE_NO_RERANK) == 0;
  const bool full = rerank && !conf_only;  // top-m by incremental merge

  const int32_t *tok = a.tok + static_cast<int64_t>(b) * D * kk;
  const float *conf = a.conf + static_cast<int64_t>(b) * D * kk;

  pdl_wait();
  if (tid == 0) {
    s_bad = 0;
    s_key[0] = tree_key(1.0f, 0, 0);  // the root: V = 1, parent field decodes to gid 0
  }
  for (int g = tid; g <= NC; g += blockDim.x) {
    s_row[g] = g == 0 ? 0 : -1;
    s_out[g] = g == 0 ? 0 : -1;
  }
  // every gid slot starts valid, so colliding ranks (only from a row that
  // repeats a token, outside the domain) never index out of range
  for (int q = tid; q < 2 * m || q < k; q += blockDim.x) {
    if (q < 2 * m) {
      s_L[q] = 0;
      s_Lg[q] = 0;
    }
    if (q < m) s_sel[q] = 0;
    if (q < k) s_E[q] = 0;
  }
  // used draft rows, row [0,0] then rows [1..D-1, *]: contiguous in the
  // input after its first k values (slot 0 = row [0,0], slot 1+(d-1)k+j =
  // row [d,j]), read in one coalesced pass; tokens and confidences outside
  // the domain are flagged and tokens clamped so the key fields stay in range
  for (int idx = tid; idx < R * k; idx += blockDim.x) {
    const int gi = idx < k ? idx : kk + (idx - k);
    int t = tok[gi];
    const float c = conf[gi];
    if (!(c >= 0.f && c <= 1.f) || t < 0 || t > 0xFFFFF) s_bad = 1;
    if (t < 0 || t > 0xFFFFF) t = 0;
    s_tok[idx] = t;
    s_conf[idx] = __fadd_rn(c, 0.0f);  // -0 -> +0: the key's unsigned order is then the float order
  }
  __syncthreads();

  // depth-1 layer: the root row's tokens (V = fl32(1 * c) = c)
  for (int r = tid; r < k; r += blockDim.x) s_key[1 + r] = tree_key(s_conf[r], 0, s_tok[r]);
  int nL = 0, cur = 0;
  for (int d = 1; d <= D; ++d) {
    __syncthreads();
    const int base = layer_base(d, k);
    const int nl = d == 1 ? k : kk;
    const uint64_t *layer = s_key + base;
    const uint64_t *L = s_L + cur * m;
    const int *Lg = s_Lg + cur * m;
    // phase A, one thread per ranked item, jobs padded to whole warps: the
    // rank of each layer key within the layer (its thread then records the
    // expansion: draft row [d, rank] for rank < k, or the no-rerank slot);
    // in the full method also each layer key against the running top-m list
    // and each list key against the layer, for the merge
    {
      const int p0 = (nl + 31) & ~31, p1 = full ? p0 : 0, p2 = full ? ((nL + 31) & ~31) : 0;
      for (int t = tid; t < p0 + p1 + p2; t += blockDim.x) {
        if (t < p0) {
          if (t < nl) {
            const int r = count_greater(layer[t], layer, nl);
            s_cnt[t] = r;
            if (r < k) {
              const int g = base + t;
              if (d < D) {
                s_E[r] = g;
                s_row[g] = d * k + r;
              }
              if (!rerank && (d - 1) * k + r < m) s_sel[(d - 1) * k + r] = g;
            }
          }
        } else if (t < p0 + p1) {
          const int it = t - p0;
          if (it < nl) s_cnt[kk + it] = count_greater(layer[it], L, nL);
        } else {
          const int it = t - p0 - p1;
          if (it < nL) s_cnt[2 * kk + it] = count_greater(L[it], layer, nl);
        }
      }
    }
    __syncthreads();
    // phase B: the merge into the other top-m buffer, and the children of
    // the expanded nodes (row [d, j] for E[j]) as the next layer
    if (full) {
      uint64_t *L2 = s_L + (cur ^ 1) * m;
      int *Lg2 = s_Lg + (cur ^ 1) * m;
      for (int q = tid; q < nl; q += blockDim.x) {
        const int pos = s_cnt[q] + s_cnt[kk + q];
        if (pos < m) {
          L2[pos] = layer[q];
          Lg2[pos] = base + q;
        }
      }
      for (int q = tid; q < nL; q += blockDim.x) {
        const int pos = q + s_cnt[2 * kk + q];
        if (pos < m) {
          L2[pos] = L[q];
          Lg2[pos] = Lg[q];
        }
      }
      nL = min(m, nL + nl);
      cur ^= 1;
    }
    if (d < D) {
      const int nbase = layer_base(d + 1, k);
      for (int q = tid; q < kk; q += blockDim.x) {
        const int j = q / k, r = q % k;
        const int p = min(max(s_E[j], 0), NC);
        const int slot = (1 + (d - 1) * k + j) * k + r;
        const float cf = s_conf[slot];
        const float v = conf_only ? cf : __fadd_rn(__fmul_rn(tkey_score(s_key[p]), cf), 0.0f);
        s_key[nbase + q] = tree_key(v, p, s_tok[slot]);
      }
    }
  }
  __syncthreads();

  // ---- selection in output order ----------------------------------------
  const int *sel = full ? (s_Lg + cur * m) : s_sel;
  if (!full && rerank && R <= 64) {
    // confidence only: best-first growth, m picks of the greatest key whose
    // parent is already in the tree.  The open candidates are the children
    // of the nodes already picked, one group per expanded node (group e: the
    // root's children for e = 0, else those of E_d[j] for e = 1+(d-1)k+j,
    // gids consecutive by child rank).  One warp holds every group's best
    // remaining child (lane e % 32, slot e / 32).  A group's children only
    // ever compete through their best, and two heads never share a parent,
    // so among heads the key order is the order of (score, 4095 - parent
    // gid), and a head is held as the 64-bit value
    //   score bits:32 | (4095 - parent gid):12 | gid:12 | (opened group + 1):7
    // (the opened group: the group a pick of this node opens, -1 if none).
    // A pick is two 32-bit warp maxima (the high word, then the low word
    // among the lanes that hold that high word), which carry the winner's
    // gid and opened group; the winner's slot and the opened group's slot
    // then take their new heads from registers.  No vote, shuffle, branch
    // or shared-memory load on a pick's critical path.
    auto first_child = [&](int e) {
      return e == 0 ? 1 : layer_base(2 + (e - 1) / k, k) + ((e - 1) % k) * k;
    };
    auto head_value = [&](int g) {
      const uint64_t key = s_key[g];
      const int row = s_row[g];
      const int opens = row >= k && 1 + row - k < R ? 1 + row - k : -1;
      const uint32_t lo = (static_cast<uint32_t>(kMaxGid - tkey_parent(key)) << 19) |
                          (static_cast<uint32_t>(g) << 7) | static_cast<uint32_t>(opens + 1);
      return (key & 0xFFFFFFFF00000000ull) | lo;
    };
    // every group's children sorted by key (rank = siblings with a greater
    // key); every slot first holds a valid value, so keys that collide (a
    // row that repeats a token, outside the domain) leave nothing out of range
    for (int q = tid; q < R * k; q += blockDim.x) s_grec[q] = head_value(first_child(q / k) + q % k);
    __syncthreads();
    for (int q = tid; q < R * k; q += blockDim.x) {
      const int e = q / k, g0 = first_child(e), g = g0 + q % k;
      const uint64_t key = s_key[g];
      int pos = 0;
      for (int r = 0; r < k; ++r) pos += s_key[g0 + r] > key;
      s_grec[e * k + pos] = head_value(g);
    }
    __syncthreads();
    if (tid < 32) {
      const int lane = tid;
      // groups lane (slot 0) and lane + 32 (slot 1): the index of the head
      // child, the head value (0: no head), the group's first child and the
      // child after the head, both held in registers so that a pick takes
      // its new head from a register (the load that refills `next` is off
      // the pick's critical path)
      const bool ok0 = lane < R, ok1 = lane + 32 < R;
      const uint64_t first0 = ok0 ? s_grec[lane * k] : 0ull, first1 = ok1 ? s_grec[(lane + 32) * k] : 0ull;
      uint64_t next0 = ok0 && k > 1 ? s_grec[lane * k + 1] : 0ull;
      uint64_t next1 = ok1 && k > 1 ? s_grec[(lane + 32) * k + 1] : 0ull;
      int n0 = 0, n1 = 0;
      uint64_t h0 = lane == 0 ? first0 : 0ull, h1 = 0ull;  // the root's group is open
      for (int pick = 0; pick < m; ++pick) {
        const uint64_t best = h0 > h1 ? h0 : h1;
        const uint32_t bhi = static_cast<uint32_t>(best >> 32), blo = static_cast<uint32_t>(best);
        const uint32_t mhi = __reduce_max_sync(0xffffffffu, bhi);
        const uint32_t mlo = __reduce_max_sync(0xffffffffu, bhi == mhi ? blo : 0u);
        // mlo == 0: no head left (cannot happen for m <= candidates, since
        // every candidate's parent is expanded); flagged, nothing moves
        const int g = static_cast<int>((mlo >> 7) & 0xFFF);
        const int e = static_cast<int>(mlo & 127) - 1;
        if (lane == 0) {
          s_sel[pick] = g;
          if (g > 0) s_out[g] = pick + 1;
          else s_bad = 1;
        }
        // the winner's group moves to its next child; a picked node that
        // was expanded opens its group (never the winner's own group)
        const uint64_t won = (static_cast<uint64_t>(mhi) << 32) | mlo;
        const bool w0 = mlo != 0 && h0 == won, w1 = mlo != 0 && h1 == won;
        const bool o0 = ok0 && e == lane, o1 = ok1 && e == lane + 32;
        if (w0) {
          h0 = next0;
          ++n0;
        }
        if (o0) {
          h0 = first0;
          n0 = 0;
        }
        if (w1) {
          h1 = next1;
          ++n1;
        }
        if (o1) {
          h1 = first1;
          n1 = 0;
        }
        if (w0 || o0) next0 = n0 + 1 < k ? s_grec[lane * k + n0 + 1] : 0ull;
        if (w1 || o1) next1 = n1 + 1 < k ? s_grec[(lane + 32) * k + n1 + 1] : 0ull;
      }
    }
  } else if (!full && rerank) {
    // confidence only with more than 64 expanded nodes: each pick is a
    // block-wide arg-max over every candidate whose parent is already in
    // the tree (s_out >= 0): thread scan, warp shuffles, then the warps'
    // winners
    __shared__ uint64_t s_wbest[kTreeThreads / 32];
    __shared__ int s_wg[kTreeThreads / 32];
    const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    for (int pick = 0; pick < m; ++pick) {
      uint64_t best = 0;
      int bg = -1;
      for (int g = 1 + tid; g <= NC; g += blockDim.x) {
        const uint64_t key = s_key[g];
        if (s_out[g] < 0 && s_out[tkey_parent(key)] >= 0 && (bg < 0 || key > best)) {
          best = key;
          bg = g;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t ob = shfl_xor_u64(best, o);
        const int og = __shfl_xor_sync(0xffffffffu, bg, o);
        if (og >= 0 && (bg < 0 || ob > best)) {
          best = ob;
          bg = og;
        }
      }
      if (lane == 0) {
        s_wbest[warp] = best;
        s_wg[warp] = bg;
      }
      __syncthreads();
      if (warp == 0) {
        best = lane < nwarps ? s_wbest[lane] : 0;
        bg = lane < nwarps ? s_wg[lane] : -1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const uint64_t ob = shfl_xor_u64(best, o);
          const int og = __shfl_xor_sync(0xffffffffu, bg, o);
          if (og >= 0 && (bg < 0 || ob > best)) {
            best = ob;
            bg = og;
          }
        }
        if (lane == 0) {
          if (bg < 0) {
            s_bad = 1;  // nothing left to add (cannot happen for m <= candidates)
            s_sel[pick] = 0;
          } else {
            s_out[bg] = pick + 1;
            s_sel[pick] = bg;
          }
        }
      }
      __syncthreads();
    }
  } else {
    for (int q = tid; q < m; q += blockDim.x) {
      const int g = sel[q];
      if (g > 0 && g <= NC) s_out[g] = q + 1;
      else s_bad = 1;
    }
  }
  __syncthreads();

  pdl_trigger();
  // ---- outputs and mask ----------------------------------------------------
  // thread (i, w): node i's fields (w == 0) and mask word w, the latter by
  // walking node i's ancestors in candidate-id space (every ancestor of a
  // selected candidate is selected; at most D+1 steps even on bad input)
  const int64_t ob = static_cast<int64_t>(b) * n;
  const int W = (n + 63) >> 6;
  for (int q = tid; q < n * W; q += blockDim.x) {
    const int i = q / W, w = q % W;
    const int src = i == 0 ? 0 : min(max(sel[i - 1], 0), NC);
    if (w == 0) {
      int t, par, dep, row;
      float sc;
      if (i == 0) {
        t = a.root_tok ? a.root_tok[b] : -1;
        par = -1; dep = 0; row = 0; sc = 1.0f;
      } else {
        const uint64_t key = s_key[src];
        t = tkey_token(key);
        sc = tkey_score(key);
        const int pg = tkey_parent(key);
        par = pg >= 0 && pg <= NC ? s_out[pg] : -1;
        if (par < 0 || par >= i) s_bad = 1;  // not closed: an input outside the domain
        dep = depth_of_gid(src, k);
        row = s_row[src];
      }
      a.node_tok[ob + i] = t;
      a.node_parent[ob + i] = par;
      if (a.node_depth) a.node_depth[ob + i] = dep;
      if (a.node_score) a.node_score[ob + i] = sc;
      if (a.node_src) a.node_src[ob + i] = src;
      if (a.node_row) a.node_row[ob + i] = row;
    }
    if (a.mask) {
      uint64_t bits = 0;
      int g = src;
      for (int steps = 0; steps <= D; ++steps) {
        const int node = s_out[g];
        if (node >= 0 && (node >> 6) == w) bits |= 1ull << (node & 63);
        if (g == 0) break;
        g = tkey_parent(s_key[g]);
        if (g < 0 || g > NC) break;
      }
      a.mask[(ob + i) * W + w] = bits;
    }
  }
  __syncthreads();
  if (tid == 0 && s_bad) report(a.status, EAGLE_ERR_INVALID);
}

__global__ void __launch_bounds__(256) tree_mask_kernel(const int32_t *parent, int n, uint64_t *mask) {
  extern __shared__ __align__(16) unsigned char smem[];
  int *s_par = reinterpret_cast<int *>(smem);
  const int b = blockIdx.x;
  const int64_t ob = static_cast<int64_t>(b) * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s_par[i] = parent[ob + i];
  __syncthreads();
  const int W = (n + 63) >> 6;
  for (int q = threadIdx.x; q < n * W; q += blockDim.x) {
    const int i = q / W, w = q % W;
    mask[(ob + i) * W + w] = mask_word(s_par, n, i, w);
  }
}

// ---- host side ---------------------------------------------------------------

size_t tree_smem_bytes(int D, int k, int m, int flags) {
  const int NC = k + (D - 1) * k * k;
  const int kk = k * k;
  size_t bytes = sizeof(uint64_t) * (NC + 1)          // s_key
               + sizeof(uint64_t) * 2 * m             // s_L
               + sizeof(int) * 2 * m                  // s_Lg
               + sizeof(int) * (2 * kk + m)           // s_cnt
               + sizeof(int) * 2 * (NC + 1)           // s_row, s_out
               + sizeof(int) * m + sizeof(int) * k    // s_sel, s_E
               + 8 * static_cast<size_t>(1 + (D - 1) * k) * k  // s_tok, s_conf
               + ((flags & EAGLE_TREE_CONFIDENCE_ONLY) ? 8 + 8 * static_cast<size_t>(1 + (D - 1) * k) * k : 0);  // s_grec
  return (bytes + 15) / 16 * 16;
}

cudaError_t launch_tree_build(const int32_t *tok, const float *conf, int B, int D, int k, int m, int flags,
                              const int32_t *root_tok, int32_t *node_tok, int32_t *node_parent,
                              int32_t *node_depth, float *node_score, int32_t *node_src,
                              int32_t *node_row, uint64_t *mask, int32_t *status, cudaStream_t st) {
  TreeArgs a;
  a.tok = tok; a.conf = conf;
  a.B = B; a.D = D; a.k = k; a.m = m; a.flags = flags;
  a.NC = k + (D - 1) * k * k;
  a.root_tok = root_tok;
  a.node_tok = node_tok; a.node_parent = node_parent; a.node_depth = node_depth;
  a.node_src = node_src; a.node_row = node_row; a.node_score = node_score;
  a.mask = mask; a.status = status;
  const size_t smem = tree_smem_bytes(D, k, m, flags);
  if (smem > 48 * 1024) {
    // the limit is raised once per device to the opt-in maximum, so it only
    // ever grows (two host threads with different sizes cannot undo each other)
    static std::atomic<unsigned long long> configured{0};
    const cudaError_t e = set_smem_limit_max_once(tree_build_kernel, configured);
    if (e != cudaSuccess) return e;
  }
  return launch_chained(tree_build_kernel, dim3(B), dim3(kTreeThreads), smem, st, a);
}

cudaError_t launch_tree_mask(const int32_t *parent, int B, int n, uint64_t *mask, cudaStream_t st) {
  tree_mask_kernel<<<B, 256, sizeof(int) * n, st>>>(parent, n, mask);
  return cudaGetLastError();
}

}  // namespace eagle
