"""Prefix groups for decode over shared blocks: which consecutive sequences of a
batch share leading KV blocks, and how many.

Test infrastructure (see the package docstring). The product's planner (C++,
in the library) is compared with this model group by group.

What the pages fix: parallel samples and beams of one prompt share the
prompt's blocks (and beams their common history) by reference to the same
physical blocks, not by copies (abeam.tech summary of "Efficient Memory
Management for Large Language Model Serving with PagedAttention", section
"並列サンプリングやビームサーチでの共有"; blog "数万トークンでもVRAMが溢れ
ない！…", "OSの知恵をGPUへ"). Two sequences whose tables hold the same
physical ids at the same leading positions therefore hold the same K and V
there, and attention over those positions can read them once for all the
queries of the group.

Readings (the pages give no kernel for it):
* full(s) = L_s // 16 blocks of sequence s are full; only full blocks are
  shared by a group (a partial block is written by its sequence next).
* common(a, b) = the number of leading table entries j < min(full(a),
  full(b)) with table[a][j] == table[b][j] >= 0.
* Greedy, in batch order: a group starts at sequence i with P = full(i) and
  takes i+1, i+2, ... while fewer than max_members are in it and
  P' = min(P, common(previous member, next)) >= min_shared; P becomes P'.
  A group of one is no group: its sequence gets prefix 0. The next group
  starts after the last member.
* Output: groups (first, count, prefix_blocks) and, per sequence, the
  prefix blocks its group shares (0 outside groups). Attention over a
  grouped sequence is then the merge of its share of the prefix pass
  (positions < 16 P) and its own suffix (positions >= 16 P).
"""

BLOCK_SIZE = 16


def full_blocks(length):
    return int(length) // BLOCK_SIZE


def common_blocks(row_a, len_a, row_b, len_b):
    n = min(full_blocks(len_a), full_blocks(len_b))
    k = 0
    while k < n and row_a[k] == row_b[k] and row_a[k] >= 0:
        k += 1
    return k


def plan_prefix_groups(tables, lens, max_members, min_shared):
    """Returns (groups, seq_prefix): groups is a list of (first, count,
    prefix_blocks); seq_prefix[s] is the prefix of s's group or 0."""
    S = len(lens)
    rows = [list(map(int, r)) for r in tables]
    seq_prefix = [0] * S
    groups = []
    i = 0
    while i < S:
        members = [i]
        P = full_blocks(lens[i])
        j = i + 1
        while j < S and len(members) < max_members:
            c = common_blocks(rows[j - 1], lens[j - 1], rows[j], lens[j])
            p_new = min(P, c)
            if p_new < min_shared:
                break
            P = p_new
            members.append(j)
            j += 1
        if len(members) >= 2:
            groups.append((i, len(members), P))
            for m in members:
                seq_prefix[m] = P
        i = j
    return groups, seq_prefix
