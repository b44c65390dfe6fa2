"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This package draws random tensors and builds paged layouts (block tables,
lengths, poison fill). It holds none of the method's arithmetic: no summary,
bound, selection, softmax or pooling is computed here.
"""
from .workloads import (  # noqa: F401
    PAGE_SIZE,
    QuestDecodeWorkload,
    QuestDecodeInputs,
    SnapKVWorkload,
    SnapKVInputs,
    TINY_QUEST_4K,
    QWEN3_4B_QUEST_32K,
    QWEN3_30B_A3B_QUEST_128K,
    SNAPKV_PREFILL_32K,
    SNAPKV_AIME_32K,
    SNAPKV_AGENT_32K,
    MLA_GLM_QUEST_32K,
    QUEST_WORKLOADS,
    make_quest_decode_inputs,
    make_snapkv_inputs,
    pages_for_tokens,
)
