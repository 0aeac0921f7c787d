/* A plain C99 program that uses the library through include/pa.h alone: the
 * host block allocator driven by a script of operations read from stdin,
 * one per line:
 *   add S | append S N | fork P C | free S
 * After each operation it prints one line: the call's status, then for an
 * append the slots it returned and the copy-on-write pair (or "-"), and
 * finally the number of free blocks.  At the end it prints every live
 * sequence's length and block table and the free list.  The test that builds
 * and runs it replays the same script on the allocator model of the block
 * manager and compares the two transcripts.
 *
 * Usage: c_abi_consumer NUM_BLOCKS BLOCK_SIZE < script
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pa.h"

#define MAX_SEQS 64
#define MAX_TOKENS 4096

int main(int argc, char **argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s NUM_BLOCKS BLOCK_SIZE < script\n", argv[0]);
        return 2;
    }
    const int num_blocks = atoi(argv[1]), block_size = atoi(argv[2]);
    pa_alloc *a = NULL;
    pa_status st = pa_alloc_create(num_blocks, block_size, NULL, &a);
    if (st != PA_OK) {
        fprintf(stderr, "create: %s\n", pa_status_string(st));
        return 1;
    }
    static int64_t slots[MAX_TOKENS];
    int live[MAX_SEQS] = {0};
    char op[16];
    long x, y;
    while (scanf("%15s %ld", op, &x) == 2) {
        if (x < 0 || x >= MAX_SEQS) return 2;
        if (strcmp(op, "add") == 0) {
            st = pa_seq_add(a, x);
            if (st == PA_OK) live[x] = 1;
            printf("add %d", (int)st);
        } else if (strcmp(op, "append") == 0) {
            if (scanf("%ld", &y) != 1 || y < 0 || y > MAX_TOKENS) return 2;
            int64_t cow[2];
            int n_cow = 0;
            st = pa_seq_append(a, x, (int)y, slots, cow, &n_cow);
            printf("append %d", (int)st);
            if (st == PA_OK) {
                printf(" slots");
                for (long i = 0; i < y; ++i) printf(" %lld", (long long)slots[i]);
                if (n_cow)
                    printf(" cow %lld %lld", (long long)cow[0], (long long)cow[1]);
                else
                    printf(" cow -");
            }
        } else if (strcmp(op, "fork") == 0) {
            if (scanf("%ld", &y) != 1 || y < 0 || y >= MAX_SEQS) return 2;
            st = pa_seq_fork(a, x, y);
            if (st == PA_OK) live[y] = 1;
            printf("fork %d", (int)st);
        } else if (strcmp(op, "free") == 0) {
            st = pa_seq_free(a, x);
            if (st == PA_OK) live[x] = 0;
            printf("free %d", (int)st);
        } else {
            return 2;
        }
        printf(" free_blocks %d\n", pa_alloc_num_free(a));
    }
    static int32_t table[MAX_TOKENS];
    for (int s = 0; s < MAX_SEQS; ++s) {
        if (!live[s]) continue;
        int64_t len = 0;
        int n = 0;
        if (pa_seq_len(a, s, &len) != PA_OK ||
            pa_seq_block_table(a, s, table, MAX_TOKENS, &n) != PA_OK)
            return 1;
        printf("seq %d len %lld table", s, (long long)len);
        for (int i = 0; i < n; ++i) printf(" %d", table[i]);
        printf("\n");
    }
    int n = 0;
    if (pa_alloc_free_list(a, table, MAX_TOKENS, &n) != PA_OK) return 1;
    printf("free_list");
    for (int i = 0; i < n; ++i) printf(" %d", table[i]);
    printf("\n");
    pa_alloc_destroy(a);
    return 0;
}
