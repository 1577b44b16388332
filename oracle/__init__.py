"""CPU oracle for the paged-KV attention hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct restatements of what each step computes, in
float64 NumPy (bit copies for the cache scatter).  Only the tests, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
anything here.  The CUDA library never links, imports or calls it, and this
package imports nothing from the CUDA package: the two share no code.

Pages cited (by title and section):

  [LIFE]  "一个 prompt 的一生：nano-vllm 从起服务到吐出 token"
          (violet-quartz.github.io) -- §2.2.3 KV cache pool, §3.3.2
          ModelRunner.run and the prepare_prefill example, §3.5 Context, §4.
  [UML]   the Nano-vLLM walk-through at uml.org.cn -- §1 "关键步骤" Step2
          (slot formula and its worked example), §2.4 Model Runner (store, then
          the prefill or decode attention op, then temperature / softmax /
          Gumbel-max sampling), §3.2 "Attention运算" (tensor formats) and
          "KV cache的写入函数" (get_slots).
  [SRC2]  "《Nano-vLLM源码逐行解析》第2篇 sequence.py、scheduler.py"
          (yeyulingfeng.com) -- the Sequence counter walkthrough (600-token
          prompt, one cached block, budget 200) and the decode-stage rule that
          a block is appended only when the last one is full.

Functions and their pins (all pins are tests under ``tests/`` marked not-gpu):

  slots.slot_of, slots.get_slots, slots.prefill_metadata, slots.decode_slot,
  slots.num_blocks, slots.last_block_num_tokens, slots.chunk_rounds
      pinned to the pages' printed values (25*4+2=102; [28 29 30 | 12 13];
      the 600/256/200 walkthrough; 600 tokens in blocks 256+256+88).
  kv_store.kv_store
      pinned by brute force on tiny pools and by the 102 example.
  attention.paged_decode, attention.paged_prefill_varlen
      pinned to a library routine (torch scaled_dot_product_attention in
      float64 on contiguous K/V), to pure-Python brute force on tiny inputs,
      to V_0 exactly when one key is visible, to gather-through-a-random-table
      == dense, to prefix-cached chunked == one-shot, and to pool-permutation
      invariance.
  sampler.sample (with sampler.sample_key_form as a second statement)
      pinned to greedy argmax when the noise is 1, to the Gumbel-max law
      P(token k) = softmax(logits/T)_k by a chi-square test, and to the
      lowest-index tie rule.

  sampler.philox4x32_10 / philox_words / philox_exp_noise / sample_philox
      the counter-based noise of the in-kernel-noise sampler: the generator
      is pinned to the published Philox4x32-10 known-answer vectors (Random123,
      Salmon et al., SC 2011); the stream built on it is checked by inverting
      its round, by output statistics, and by the Gumbel-max law of its draws.

Every function is pinned.
"""
from . import attention, kv_store, sampler, slots  # noqa: F401
