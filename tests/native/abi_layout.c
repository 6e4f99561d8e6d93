/* Prints the size and field offsets of the ABI structs as "name offset"
 * lines, for the comparison with the Python binding's ctypes structures. */
#include <stddef.h>
#include <stdio.h>

#include "attn_bwd.h"

#define FIELD(T, f) printf(#T "." #f " %zu\n", offsetof(T, f))

int main(void) {
  printf("attn_problem_t %zu\n", sizeof(attn_problem_t));
  FIELD(attn_problem_t, B);
  FIELD(attn_problem_t, Hq);
  FIELD(attn_problem_t, Hk);
  FIELD(attn_problem_t, Sq);
  FIELD(attn_problem_t, Sk);
  FIELD(attn_problem_t, D);
  FIELD(attn_problem_t, scale);
  FIELD(attn_problem_t, q_stride);
  FIELD(attn_problem_t, k_stride);
  FIELD(attn_problem_t, v_stride);
  FIELD(attn_problem_t, o_stride);
  FIELD(attn_problem_t, do_stride);
  FIELD(attn_problem_t, flags);
  FIELD(attn_problem_t, cu_seqlens_q);
  FIELD(attn_problem_t, cu_seqlens_k);
  FIELD(attn_problem_t, total_q);
  FIELD(attn_problem_t, total_k);
  printf("attn_mask_t %zu\n", sizeof(attn_mask_t));
  FIELD(attn_mask_t, window_left);
  FIELD(attn_mask_t, window_right);
  FIELD(attn_mask_t, num_sink);
  FIELD(attn_mask_t, bottom_right);
  printf("attn_sparse_t %zu\n", sizeof(attn_sparse_t));
  FIELD(attn_sparse_t, ori_kv);
  FIELD(attn_sparse_t, cmp_kv);
  FIELD(attn_sparse_t, cmp_idx);
  FIELD(attn_sparse_t, n_ori);
  FIELD(attn_sparse_t, n_cmp);
  FIELD(attn_sparse_t, topk);
  FIELD(attn_sparse_t, ori_win_left);
  FIELD(attn_sparse_t, ori_win_right);
  FIELD(attn_sparse_t, d_ori_kv);
  FIELD(attn_sparse_t, d_cmp_kv);
  FIELD(attn_sparse_t, cmp_ratio);
  return 0;
}
