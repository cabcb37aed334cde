"""CPU fp64 oracle of the GQA decode step.

Test infrastructure: imported only by the tests, the smoke check and the
benchmark's CPU-baseline / reference legs. The product path never imports it.
"""
