"""The prefix-grouping rule of the block manager, written out over an oracle
manager's tables, for exact comparison with the library's bm_prefix_groups."""
import numpy as np


def expected_groups(o, ids, maxm):
    """The grouping rule written out over the oracle's tables: buckets by first
    block in order of their first member, cut into consecutive runs of maxm;
    a run with 2+ members and a common full prefix of 1+ blocks is a group."""
    buckets = {}
    for i, sid in enumerate(ids):
        if o.tables[sid]:
            buckets.setdefault(o.tables[sid][0], []).append(i)
    members, prefix, blocks = [], [], []
    seq_group = [-1] * len(ids)
    for mem in buckets.values():                     # dicts keep insertion order
        for c in range(0, len(mem), maxm):
            run = mem[c:c + maxm]
            tabs = [o.tables[ids[i]] for i in run]
            full = min(o.lens[ids[i]] // o.block_size for i in run)
            pre = 0
            while pre < full and all(t[pre] == tabs[0][pre] for t in tabs):
                pre += 1
            if len(run) < 2 or pre < 1:
                continue
            for i in run:
                seq_group[i] = len(members)
            members.append(run + [-1] * (maxm - len(run)))
            prefix.append(pre)
            blocks.append(pre + sum(len(t) - pre for t in tabs))
    return members, prefix, seq_group, blocks


def assert_groups_exact(o, ids, maxm, got):
    exp = expected_groups(o, ids, maxm)
    assert [np.asarray(x).tolist() for x in got] == [list(x) for x in exp]
