// Verification walk over the kept tree ("EAGLE-3 精读" §5 正确性、复现与风险:
// with the target's standard verifier, greedy keeps the target's sequence and
// sampling keeps its distribution when the residual correction is done).
//
// Greedy: from the root, descend into the child whose token is the target's
// argmax at the current node; stop when no child matches; the argmax at the
// stop node is the bonus token.
//
// Sampling: the tree's children are deterministic top-k picks, i.e. point-mass
// proposals, so the exact acceptance rule is: child c_i (canonical order) is
// accepted iff U_i (1 - R) < p(c_i), where p = softmax(z / T) and R is the
// target mass of the children already rejected at this node; when none is
// accepted (or the node is a leaf) the bonus token is the Gumbel-argmax of z/T
// over the node's non-children, an exact draw from the residual distribution.
// One thread per request; all per-node quantities come from the target head.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "philox.cuh"

namespace e3 {

__global__ void walk_kernel(WalkArgs a) {
  pdl_begin();
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.B) return;
  const unsigned long long rid = a.round_ptr ? *a.round_ptr : a.round_id;
  const size_t tb = (size_t)b * a.M1;
  int u = 0, n = 0;
  int* path = a.path + (size_t)b * a.D;
  int* out = a.out_tokens + (size_t)b * (a.D + 1);
  for (int i = 0; i < a.D; ++i) path[i] = -1;
  for (int i = 0; i <= a.D; ++i) out[i] = -1;
  while (true) {
    const size_t r = tb + u;
    int nc = a.n_child[r];
    int next = -1;
    if (!a.sampling) {
      int tgt = a.z_arg[r];
      for (int i = 0; i < nc; ++i) {
        int c = a.child_node[r * a.kmax + i];
        if (a.t_tok[tb + c] == tgt) { next = c; break; }
      }
    } else {
      float lse = a.lse[r], rej = 0.f;
      for (int i = 0; i < nc; ++i) {
        float p = expf(a.child_z[r * a.kmax + i] * a.inv_t - lse);
        float U = verify_uniform(a.seed, rid, b, u, i);
        if (U * (1.f - rej) < p) { next = a.child_node[r * a.kmax + i]; break; }
        rej += p;
      }
    }
    if (next < 0 || n >= a.D) {
      out[n] = a.sampling ? a.g_arg[r] : a.z_arg[r];
      break;
    }
    path[n] = next;
    out[n] = a.t_tok[tb + next];
    ++n;
    u = next;
  }
  a.accept_len[b] = n;
}

void launch_walk(const WalkArgs& a, cudaStream_t st) {
  launch_pdl(walk_kernel, dim3((a.B + 63) / 64), dim3(64), 0, st, a);
}

__global__ void set_u64_kernel(unsigned long long* p, unsigned long long v) { pdl_begin(); *p = v; }

void launch_set_u64(unsigned long long* p, unsigned long long v, cudaStream_t st) {
  launch_pdl(set_u64_kernel, dim3(1), dim3(1), 0, st, p, v);
}

}  // namespace e3
