"""CPU oracle for the block-quantized int4 x int8 product.

TEST INFRASTRUCTURE ONLY: the product library never imports this package.
"""
