/* A plain C client of libpagedkv: the host block manager driven through the C
 * ABI alone (no Python, no torch), printing what it hands out so a test can
 * compare it with the CPU oracle. Build: cc -I include this.c -L<dir> -lpagedkv */
#include <stdint.h>
#include <stdio.h>

#include "pagedkv.h"

static int check(int st, const char* what) {
    if (st != PKV_OK) printf("error %s %d %s\n", what, st, pkv_status_string(st));
    return st;
}

static void table(pkv_block_manager* bm, int64_t sid) {
    int32_t t[16];
    int n = 0;
    check(bm_block_table(bm, sid, t, 16, &n), "bm_block_table");
    printf("table %lld", (long long)sid);
    for (int i = 0; i < n; ++i) printf(" %d", t[i]);
    printf("\n");
}

int main(void) {
    const int32_t order[12] = {5, 2, 7, 0, 3, 6, 1, 4, 11, 9, 10, 8};
    pkv_block_manager* bm = bm_create(12, 4, order, 12);
    if (!bm) {
        printf("error bm_create\n");
        return 1;
    }
    /* sequence 0: 6 tokens (two blocks, the second half full) */
    check(bm_add_seq(bm, 0), "bm_add_seq");
    for (int i = 0; i < 6; ++i) {
        int64_t slot;
        int32_t s, d;
        check(bm_append_slot(bm, 0, &slot, &s, &d), "bm_append_slot");
        printf("slot 0 %lld cow %d %d\n", (long long)slot, s, d);
    }
    /* fork: 1 shares both blocks; its next token copies the partial one */
    check(bm_fork(bm, 0, 1), "bm_fork");
    for (int64_t sid = 1; sid >= 0; --sid) {
        int64_t slot;
        int32_t s, d;
        check(bm_append_slot(bm, sid, &slot, &s, &d), "bm_append_slot");
        printf("slot %lld %lld cow %d %d\n", (long long)sid, (long long)slot, s, d);
    }
    table(bm, 0);
    table(bm, 1);
    /* a beam step: two new beams both continue sequence 1, then 0 and 1 go */
    const int64_t old_ids[2] = {0, 1}, new_ids[2] = {2, 3};
    const int32_t parents[2] = {1, 1};
    check(bm_beam_step(bm, old_ids, 2, parents, new_ids, 2), "bm_beam_step");
    table(bm, 2);
    table(bm, 3);
    int32_t freel[12];
    const int nf = bm_free_list(bm, freel, 12);
    printf("free");
    for (int i = 0; i < nf; ++i) printf(" %d", freel[i]);
    printf("\n");
    /* a decode step over both beams: 2 copies the shared partial block, which
     * leaves 3 its only owner, so 3 writes in place */
    const int64_t step_ids[2] = {2, 3};
    int64_t slots[2], pairs[4];
    int ncow = 0;
    check(bm_append_slots(bm, step_ids, 2, slots, pairs, &ncow), "bm_append_slots");
    printf("step %lld %lld", (long long)slots[0], (long long)slots[1]);
    for (int i = 0; i < ncow; ++i)
        printf(" cow %lld %lld", (long long)pairs[2 * i], (long long)pairs[2 * i + 1]);
    printf("\n");
    /* a chunk the pool cannot hold is refused whole: nothing changes */
    const int free_before = bm_num_free(bm);
    int len_before = 0, len_after = 0;
    check(bm_seq_len(bm, 2, &len_before), "bm_seq_len");
    const int st = bm_append_n(bm, 2, 4 * (free_before + 1), pairs, 2, &ncow);
    check(bm_seq_len(bm, 2, &len_after), "bm_seq_len");
    printf("refused %d cow %d len %d %d free %d %d\n", st, ncow, len_before, len_after,
           free_before, bm_num_free(bm));
    /* an unknown sequence is an error, and the manager is unchanged */
    printf("unknown %d\n", bm_free_seq(bm, 99));
    bm_destroy(bm);

    /* prefix caching and swapping on a second manager: a 9-token prompt is
     * served, a second request reuses its two full blocks, then the first
     * request is swapped out and back in */
    const int32_t order2[8] = {0, 1, 2, 3, 4, 5, 6, 7};
    pkv_block_manager* pc = bm_create(8, 4, order2, 8);
    if (!pc) {
        printf("error bm_create\n");
        return 1;
    }
    check(bm_enable_prefix_caching(pc), "bm_enable_prefix_caching");
    check(bm_set_host_blocks(pc, 4), "bm_set_host_blocks");
    const int32_t prompt[9] = {5, 6, 7, 8, 9, 10, 11, 12, 13};
    int cached = -1;
    check(bm_add_seq_prompt(pc, 0, prompt, 9, &cached), "bm_add_seq_prompt");
    int64_t pslots[9], ppairs[4];
    int pcow = 0;
    check(bm_append_tokens(pc, 0, prompt + cached, 9 - cached, pslots, ppairs, 2, &pcow),
          "bm_append_tokens");
    printf("prompt 0 cached %d", cached);
    for (int i = 0; i < 9 - cached; ++i) printf(" %lld", (long long)pslots[i]);
    printf("\n");
    check(bm_add_seq_prompt(pc, 1, prompt, 9, &cached), "bm_add_seq_prompt");
    printf("prompt 1 cached %d\n", cached);
    int64_t hits = 0, looks = 0;
    int ncached = 0, nev = 0;
    check(bm_cache_stats(pc, &hits, &looks, &ncached, &nev), "bm_cache_stats");
    printf("stats %lld %lld %d %d\n", (long long)hits, (long long)looks, ncached, nev);
    int64_t sp[8];
    int nsp = 0;
    check(bm_swap_out(pc, 0, sp, 4, &nsp), "bm_swap_out");
    printf("out");
    for (int i = 0; i < nsp; ++i) printf(" %lld %lld", (long long)sp[2 * i], (long long)sp[2 * i + 1]);
    printf("\n");
    check(bm_swap_in(pc, 0, sp, 4, &nsp), "bm_swap_in");
    printf("in");
    for (int i = 0; i < nsp; ++i) printf(" %lld %lld", (long long)sp[2 * i], (long long)sp[2 * i + 1]);
    printf("\n");
    bm_destroy(pc);
    return 0;
}
