"""CPU oracle for causal GQA flash attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU baseline import this
package. The product path (``causal_gqa_flash_attn_gb300``) never does.
"""
