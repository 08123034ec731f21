// Host driver for fsdp_emulated_ranks_gb300/csrc/reducer_state.h.  Reads
// scenarios from stdin and prints, per mark, the status and the buckets it
// made launchable, so the test can compare them with its own model.
//   input:  S, then per scenario: T B, T bucket ids, M, M tensor indices
//           (-9 means "reset the iteration")
//   output: per mark one line "rc launched | b0 b1 ..."; "reset" lines.
#include <cstdio>
#include <vector>

#include "reducer_state.h"

int main() {
  int S = 0;
  if (scanf("%d", &S) != 1) return 2;
  for (int s = 0; s < S; ++s) {
    int T = 0, B = 0, M = 0;
    if (scanf("%d %d", &T, &B) != 2) return 2;
    std::vector<int> tb(T > 0 ? T : 1);
    for (int t = 0; t < T; ++t)
      if (scanf("%d", &tb[t]) != 1) return 2;
    cr::ReducerState st(tb.data(), T, B);
    if (scanf("%d", &M) != 1) return 2;
    printf("scenario %d complete=%d\n", s, st.complete() ? 1 : 0);
    for (int i = 0; i < M; ++i) {
      int t = 0;
      if (scanf("%d", &t) != 1) return 2;
      if (t == -9) {
        st.reset();
        printf("reset\n");
        continue;
      }
      std::vector<int> launch;
      const int rc = st.mark(t, &launch);
      printf("%d %d %d |", rc, st.launched(), st.complete() ? 1 : 0);
      for (int b : launch) printf(" %d", b);
      printf("\n");
    }
  }
  return 0;
}
