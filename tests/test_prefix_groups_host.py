"""The prefix-group rule of splash_verify_attention_shared on hand-derived
cases (the model the GPU tests compare the device plan with)."""
from __future__ import annotations

import pytest

from common import expected_group_plan as plan
from speculative_verify_attention_kv_gb300 import workloads as wl


def test_four_sequences_of_96_rows_take_three_blocks():
    # 4 x (24576 + 8192) keys, T = 16, G = 6: rows 384 -> 3 blocks of 128;
    # per KV head 3 x 384 prefix tiles + 4 x (513 - 384) own tiles
    W = wl.make("shared_prefix")
    ctx = [int(x) for x in W.context_lens]
    T = [int(x) for x in W.block_lens]
    assert plan(ctx, T, list(W.shared_lens()), 6, 4) == (7, 4 * (3 * 384 + 4 * 129))
    # without links every sequence reads all 513 of its tiles
    assert plan(ctx, T, [0] * 4, 6, 4) == (4, 4 * 4 * 513)


def test_single_token_blocks_share_one_block():
    # 4 x 6 rows fit one block: the 1984-key prefix (31 tiles) is read once
    ctx, T = [2000, 2100, 2050, 2300], [1, 1, 1, 1]
    items, tiles = plan(ctx, T, [0, 1984, 1984, 1984], 6, 1)
    own = sum(-(-(c + t) // 64) - 31 for c, t in zip(ctx, T))
    assert (items, tiles) == (5, 31 + own)


def test_full_row_blocks_are_not_stacked():
    # 128 rows per sequence: as many blocks as sequences, so no group
    assert plan([400, 500], [16, 16], [0, 320], 8, 2) == (2, 2 * (7 + 9))


@pytest.mark.parametrize("link", [0, 1, 63])
def test_links_below_a_tile_make_no_group(link):
    assert plan([300, 300], [4, 4], [0, link], 6, 1) == (2, 5 + 5)


def test_an_idle_sequence_breaks_the_run():
    assert plan([300, 300, 300], [4, 0, 4], [0, 256, 256], 6, 1) == (3, 5 + 5)


def test_prefix_is_the_smallest_link_cut_to_contexts_and_a_tile():
    # links 512 and 200 -> 200 -> 192 keys (3 tiles); rows 24 + 48 + 6 -> 1 block
    ctx, T = [600, 700, 512], [4, 8, 1]
    items, tiles = plan(ctx, T, [0, 512, 200], 6, 1)
    own = sum(-(-(c + t) // 64) - 3 for c, t in zip(ctx, T))
    assert (items, tiles) == (4, 3 + own)
    # a link past a context is cut to it: the 208-key context bounds the prefix
    assert plan([208, 300], [1, 1], [0, 10 ** 6], 6, 1)[0] == 3


def test_two_groups_number_their_blocks_after_the_sequences():
    ctx, T = [600, 700, 512, 900, 1000, 530], [4, 8, 1, 16, 2, 3]
    items, _ = plan(ctx, T, [0, 512, 512, 0, 200, 512], 6, 4)
    assert items == 6 + 2
